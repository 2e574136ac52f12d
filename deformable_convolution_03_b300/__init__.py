"""B300-native (sm_103a) DCNv3 / DCNv4 core deformable aggregation.

The computation lives in ``libdcn_b300.so`` (CUDA, built by :mod:`.build`);
:mod:`.binding` is its ctypes binding.  Importing this package does not load
the library: the first call does, and raises if it has not been built.
"""
from .binding import (  # noqa: F401
    DCN_BF16, DCN_F16, DCN_F32, DCNError, Params, center_feature_scale,
    center_feature_scale_backward, core_bwd, core_fwd, dcn_core, dcn_core_bwd,
    dcn_core_bwd_workspace, dcn_core_fwd, dcn_num_points, dcn_out_shape, dcn_status_str,
    dcn_version, dwconv_ln_gelu, linear)
