"""Paged KV cache hot path for NVIDIA GB300 (sm_103a).

The work happens in ``libpa.so`` (hand-written CUDA kernels and a C++ host
block manager, C ABI in ``include/pa.h``); this package is its binding.
"""
from .api import (  # noqa: F401
    PA_BF16, PA_ERR_CUDA, PA_ERR_INVALID_ARG, PA_ERR_NOT_FOUND, PA_ERR_OUT_OF_BLOCKS,
    PA_ERR_TIMEOUT, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_F16, PA_F32, PA_OK, BlockManager, PAError,
    pa_check_wait_timeout, pa_compute_slot_mapping, pa_copy_blocks, pa_decode, pa_decode_append, pa_decode_contiguous, pa_decode_plan,
    pa_decode_shared_prefix,
    pa_decode_shared_prefix_workspace_size, pa_decode_splitk, pa_decode_static_scratch, pa_decode_workspace_size,
    pa_device_status, pa_lse_merge, pa_reshape_and_cache, pa_swap_blocks,
)
from ._lib import library_path, load as load_library  # noqa: F401
