"""GB300 (sm_103a) depthwise causal short convolution with fused SiLU.

The computation lives in ``libcconv.so`` (C ABI: ``include/cconv.h``); this package is its
thin Python binding with the same names, plus the build step and the seeded synthetic
input generators.  Importing the package does not load the library; the first call does,
and raises if it has not been built.
"""
from .autograd import causal_conv1d  # noqa: F401
from .binding import (  # noqa: F401
    CCONV_ACT_NONE,
    CCONV_ACT_SILU,
    CCONV_BF16,
    CCONV_F32,
    IDX_DUPLICATE,
    IDX_NEGATIVE,
    IDX_OUT_OF_RANGE,
    CConvError,
    cconv_bwd,
    cconv_bwd_multi,
    cconv_bwd_multi_workspace_bytes,
    cconv_bwd_noalloc,
    cconv_bwd_varlen,
    cconv_bwd_varlen_workspace_bytes,
    cconv_bwd_workspace_bytes,
    cconv_device_fault,
    cconv_fwd,
    cconv_fwd_multi,
    cconv_fwd_varlen,
    cconv_status_str,
    cconv_update,
    cconv_update_ex,
    describe,
    header_functions,
    lib_path,
    load,
)
