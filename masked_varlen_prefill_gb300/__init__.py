"""Masked varlen prefill attention for GB300 (sm_103a).

Thin Python binding over the C-ABI library ``lib/libmvp.so`` (declared in
``include/mvp.h``).  The functions below only marshal arguments (torch CUDA
tensors -> device pointers, sizes, the current stream) and raise on a non-zero
status; every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: if the library is missing, importing the binding's
functions raises.
"""

from ._lib import (  # noqa: F401
    MVP_ERR_ARG,
    MVP_ERR_CAPACITY,
    MVP_ERR_CUDA,
    MVP_ERR_DEVICE_BOUNDS,
    MVP_ERR_DEVICE_TIMEOUT,
    MVP_ERR_UNSUPPORTED,
    MVP_OK,
    FAULT_NONE,
    FAULT_WITHHOLD_PROBS,
    SINK_KEY0_BIAS,
    SINK_NONE,
    SINK_NULL_LOGIT,
    VARIANT_D512_HEAD_SPLIT,
    VARIANT_DEFAULT,
    AttnOptions,
    MvpError,
    StepMetadata,
    attn_accounting,
    attn_fwd_varlen,
    attn_fwd_paged,
    attn_fwd_varlen_host,
    attn_fwd_varlen_scan,
    attn_fwd_varlen_static_ws,
    attn_workspace_size,
    bounds_checked,
    fill_query_ranges,
    get_last_device_error,
    last_launch_count,
    library_path,
    load_library,
    meta_block_layout,
    meta_pack,
)
