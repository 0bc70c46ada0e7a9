"""Exact attention on one GB300 GPU: FlashAttention-2-style forward, three-kernel
backward and split-KV flash decoding, as hand-written sm_103a CUDA behind the
C ABI in include/fa.h (libfa.so, built in-tree by ``exact_attention_gb300.build``).

The library is loaded on first use; if it has not been built, every call raises.
"""
from ._binding import (  # noqa: F401
    EXPORTS,
    FA_BF16,
    FA_ERR_CUDA,
    FA_ERR_INVALID,
    FA_ERR_TIMEOUT,
    FA_ERR_UNSUPPORTED,
    FA_F16,
    FA_F32,
    FA_OK,
    FAError,
    backward,
    decode,
    fa_bwd,
    fa_bwd_workspace_bytes,
    fa_decode,
    fa_decode_static,
    fa_decode_ex,
    fa_fwd_host,
    fa_bwd_ws,
    fa_bwd_ws_workspace_bytes,
    fa_fwd_host_workspace_bytes,
    fa_decode_ex_workspace_bytes,
    fa_debug_inject,
    fa_decode_workspace_bytes,
    fa_fwd,
    fa_fwd_workspace_bytes,
    fa_fwd_ws,
    fa_last_error_message,
    fa_last_status,
    fa_set_wait_budget_ns,
    fa_status_string,
    forward,
    forward_workspace,
    lib,
    split_workspace,
)
