"""Split-KV (Flash-Decoding) single-token decode attention for GB300 (sm_103a).

A thin ctypes binding over ``libfd.so`` (C ABI in ``include/fd.h``).  Every step of
the computation runs in the library's CUDA kernels; this module only marshals torch
tensors into ``fd_tensor`` descriptors, passes the current CUDA stream, and turns
status codes into exceptions.  There is no CPU fallback: if the library is missing
or fails to load, every call raises.
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    FD_MERGE_IN_KERNEL, FD_MERGE_KERNEL, FD_PATH_AUTO, FD_PATH_MMA, FD_PATH_SIMT, FD_PATH_TCGEN05,
    FD_FROM_PROCESS, FD_SCHEDULE_AUTO, FD_SCHEDULE_GRID, FD_SCHEDULE_HEAD_GROUPS,
    FD_SCHEDULE_PERSISTENT, FD_SCHEDULE_TAIL_SHARING, FdError, FdOptions,
    Plan, decode_attention, decode_attention_fp8kv, decode_attention_noalloc,
    decode_partial, decode_partial_fp8kv, get_merge_mode, get_path, get_schedule, lib, library_path, merge_partials,
    num_splits_for_lengths, num_splits_heuristic, options, partial_kernel_name, partial_kernel_name_for,
    read_device_error,
    resolve_num_splits, selftest_bounded_wait, selftest_stalled_decode,
    set_merge_mode, set_path, set_schedule, workspace_init, workspace_partials, workspace_size,
)
