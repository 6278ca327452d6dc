"""GB300-native LongFlow decode step.

One call performs the fused per-step operator of "LongFlow: Efficient KV Cache
Compression for Reasoning Models": it writes the current token's K/V into the
slot chosen at the previous step, runs decode attention over the static,
mask-gated cache, computes LongFlowScore for every live slot and returns the
argmin slot to overwrite next. The work runs in the CUDA kernels of
``lib/liblf_decode.so`` (C ABI in ``include/lf_decode.h``). This package only
binds it (``_binding``), builds it (``build``) and describes the synthetic
workloads (``workloads``).
"""
from ._binding import (  # noqa: F401
    EXPORTED, KERNEL_NAMES, LF_DEVERR_BAD_WRITE_SLOT, LF_DEVERR_WAIT_TIMEOUT,
    LF_ERR_CUDA, LF_ERR_INVALID_ARG, LF_ERR_NO_MEMORY, LF_ERR_UNSUPPORTED,
    LF_KERNEL_ATTENTION, LF_KERNEL_DECODE_STEP, LF_KERNEL_SCORE, LF_MAX_TOPK, LF_OK,
    LF_STEP_FILL_EMPTY_FIRST, LF_STEP_LOG2_SCORES, LF_STEP_MASK_EVICTED, LFError, PreparedStep,
    decode_attention,
    decode_step, decode_step_ex,
    decode_step_host, decode_step_noalloc,
    decode_step_scores, device_errors, library_path, load_library, profile_collect,
    profile_enable, release_workspace, status_string, step_plan, version)
