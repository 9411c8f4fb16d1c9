"""GB300 (sm_103a) attention hot path for bounded generation.

Packed variable-length causal GQA prefill, shared-prefix beam decode attention
with parent-index suffix reorder, and two-stage beam candidate selection, as
hand-written CUDA kernels behind the C ABI in ``include/slm_attn.h``.  The
functions below are a thin marshalling layer over that library; the library
must be built (``python -m attention_packed_varlen_gb300.build``) and there is
no CPU fallback.
"""
from ._binding import (  # noqa: F401
    SlmError,
    load,
    slm_abi_version,
    slm_beam_select,
    slm_beam_select_workspace_size,
    slm_check_status,
    slm_packed_prefill_attn,
    slm_packed_prefill_attn_f32,
    slm_prefill_workspace_size,
    slm_set_wait_timeout_ns,
    slm_shared_prefix_decode_attn,
    slm_shared_prefix_decode_attn_f32,
    slm_shared_prefix_decode_workspace_size,
)
