"""Split-K paged-attention decode for GB300 (sm_103a).

The compute lives in ``libpa_decode.so`` (CUDA C++, C ABI in
``include/pa_decode.h``); this package is its thin Python binding.  Build
the library with :func:`paged_kv_decode_v2_gb300.build.build`.
"""
from ._lib import (  # noqa: F401
    LIB_PATH, PA_BF16, PA_ERR_CUDA, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE,
    PA_F16, PA_OK, PA_STATUS_BAD_BLOCK_ID, PA_STATUS_BAD_SEQ_LEN, PA_STATUS_TIMEOUT,
    PagedAttentionError, alloc_counters, alloc_workspace, load, num_partitions, pa_decode, pa_decode_choose,
    pa_decode_mq, pa_decode_mq_choose, pa_decode_mq_partition,
    pa_decode_v1, pa_decode_v1_mq, pa_decode_v2, pa_decode_v2_fused, pa_decode_v2_mq,
    pa_decode_v2_phase1,
    pa_decode_v2_phase2, pa_decode_v2_static,
    pa_selftest_wait_timeout, pa_set_launch_config, pa_set_merge_form, pa_set_rows_kernel, status_string,
    workspace_bytes)
