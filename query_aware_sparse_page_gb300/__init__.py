"""Query-aware sparse-page decode attention for GB300 (sm_103a).

The computation lives in libspg.so (hand-written CUDA, C ABI declared in
include/spg.h); this package is its ctypes binding plus device-buffer
helpers that only allocate (with torch) and never compute.
"""

from .binding import (  # noqa: F401
    BF16, DEVERR_PAGE_ID, DEVERR_SEL, DEVERR_SEQ_LEN, DEVERR_TIMEOUT, F16, I8, LIB, LIB_PATH,
    SEL_ALL, SEL_QUEST, SEL_SKETCH_INT4, SpgError, dense_decode_attention, make_params,
    sparse_decode_attention, sparse_decode_select_attend, sparse_decode_step, sparse_page_meta_update,
    sparse_page_score, sparse_page_select, sparse_page_sketch_dots, spg_abi_version, spg_clear_device_error, spg_params,
    spg_read_device_error, spg_status_str, spg_test_withhold_first_stage, spg_validate, spg_workspace_size, status_str,
    STEP_KERNEL_AUTO, STEP_KERNEL_CLUSTER, STEP_KERNEL_SCHED, spg_prefer_dense, spg_set_step_kernel, spg_step_kernel,
    spg_step_launches, step_kernel_name, step_launch_count,
)
from .buffers import DecodeBuffers, alloc_buffers, params_for  # noqa: F401
