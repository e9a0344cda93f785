"""Orthros attention hot path on GB300: Python binding of liborthros_attn.so.

The binding only marshals arguments (torch tensors -> device pointers, sizes,
the current CUDA stream) into the C ABI declared in include/orthros_attn.h.
Every step of the computation runs in the library's CUDA kernels; there is no
CPU or PyTorch fallback. If the compiled library is missing, importing the
binding still works but every call raises.
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    OrthrosError,
    lib_path,
    load_library,
    orthros_check,
    orthros_decode,
    orthros_decode_static,
    orthros_decode_workspace_size,
    orthros_extend,
    orthros_extend_workspace_size,
    orthros_last_error,
    orthros_merge_partials,
    orthros_prefill,
    orthros_prefill_backward,
    orthros_prefill_backward_workspace_size,
    orthros_prefill_from_host,
    orthros_prefill_from_host_workspace_size,
    orthros_prefill_shard,
    orthros_prefill_shard_workspace_size,
    orthros_prefill_workspace_size,
    orthros_profile_begin,
    orthros_qkv_project,
    orthros_selftest_wait_timeout,
    orthros_profile_end,
    orthros_status_string,
)
