"""Unified paged varlen flash attention (forward) for GB300 / sm_103a.

The computation lives in ``libua.so`` (hand-written CUDA behind the C ABI of
``include/ua.h``).  This package is a thin ctypes binding with the same entry
point names; it only marshals torch tensors (device memory, streams) into that
ABI.  There is no fallback: if the library is missing, every entry point raises.

Build the library with ``python -m paged_varlen_flash_gb300.build`` (or
``__graft_entry__.build()``).
"""
from .binding import (  # noqa: F401
    UA_FLAG_ALIBI, UA_FLAG_CAUSAL, UA_FLAG_SINKS, UA_FLAG_SOFTCAP, UA_FLAG_WINDOW,
    UA_FLAG_QQ_BIAS,
    UA_DEVERR_BLOCK_ID, UA_DEVERR_BOUNDS, UA_DEVERR_CONTEXT, UA_DEVERR_CU_SEQLENS,
    UA_DEVERR_TIMEOUT, UA_PATH_AUTO, UA_PATH_SPLIT_KV, UA_PATH_TENSOR_CORE, UA_PATH_DECODE_TC,
    UA_DTYPE_BF16, UA_DTYPE_FP8_E4M3, UA_PARTIALS_F32, UA_PARTIALS_BF16,
    UAError, Problem, flags_of, lib_path, load_library,
    ua_check_device_error, ua_destroy, ua_forward, ua_forward_host, ua_forward_noalloc,
    ua_forward_topk,
    ua_problem_create, ua_set_qq_bias,
    ua_status_string)
