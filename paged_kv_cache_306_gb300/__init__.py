"""GB300-native paged-attention decode.

A small C-ABI library (``_build/libpa.so``, sources in ``csrc/``, interface in
``include/pa.h``) with hand-written sm_103a kernels for the two directions of a
paged KV cache: the write path (``pa_reshape_and_cache``, ``pa_copy_blocks``)
and decode attention over the block pool (``pa_decode``), with an FP8 E4M3
cache variant of both (``pa_reshape_and_cache_scaled``, ``pa_decode_scaled``), the
three fused into one generation step (``pa_decode_step``), chunked prefill
(``pa_prefill``) and the host-side block manager that produces block tables, slots and copy-on-write
pairs (``BlockManager``, ``include/pa_block_manager.h``).  This package is the
thin Python binding; PyTorch supplies device memory and streams only.
"""
from ._binding import (  # noqa: F401
    DEVICE_ERRORS,
    BlockManager,
    LIB_PATH,
    PA_BF16,
    PA_ERR_ALIGNMENT,
    PA_ERR_CUDA,
    PA_ERR_INVALID_ARG,
    PA_ERR_OUT_OF_BLOCKS,
    PA_ERR_UNSUPPORTED,
    PA_ERR_WORKSPACE,
    PA_F16,
    PA_F32,
    PA_FP8_E4M3,
    PA_OK,
    PARTITION_AUTO,
    PARTITION_NONE,
    PAError,
    load,
    pa_copy_blocks,
    pa_decode,
    pa_decode_scaled,
    pa_decode_shared,
    pa_decode_shared_workspace_size,
    pa_decode_step,
    pa_decode_step_scaled,
    pa_decode_plan_partition,
    pa_decode_workspace_size,
    pa_get_device_error,
    pa_prefill,
    pa_launch_count,
    pa_reshape_and_cache,
    pa_set_test_wait_limit,
    pa_reshape_and_cache_scaled,
)
