"""Orthros per-layer attention operator on one GB300 (sm_103a).

A thin binding over the C ABI in ``include/orthros.h`` (``liborthros.so``):
argument marshalling only -- every step of the operator runs in the library's
CUDA kernels.  PyTorch provides device memory and the current stream.

* :func:`swa_fwd`      -- base-stream sliding-window attention, Eq. (4)
* :func:`swa_fwd_rows` -- the same for a range of output rows (chunked prefill)
* :func:`swa_fwd_lse`  -- the same with each row's log-sum-exp (for the gradient)
* :func:`xattn_fwd`    -- output-copy full causal cross-attention, Eq. (5) (optionally with
  each copy row's log-sum-exp)
* :func:`prefill_fwd`  -- both of them for one prefill layer in one call
* :func:`decode_step`  -- one fused decode step with KV-cache append
* :func:`swa_bwd`      -- gradient of the base stream (Eq. (4) and its scale-offset)
* :func:`xattn_bwd`    -- gradient of the output copies (Eq. (5)), added into dK / dV
* :func:`attn_bwd`     -- both streams' gradient of a layer in one call, dK / dV written once

If the library is missing these functions raise; there is no fallback.
"""
from ._binding import (  # noqa: F401
    DEVERR_CACHE_FULL,
    DEVERR_POSITION,
    DEVERR_RANGE,
    DEVERR_TIMEOUT,
    OrthrosError,
    attn_bwd,
    attn_bwd_workspace_size,
    decode_step,
    decode_workspace_size,
    lib,
    library_path,
    prefill_fwd,
    prefill_workspace_size,
    swa_bwd,
    swa_bwd_workspace_size,
    swa_fwd,
    swa_fwd_lse,
    swa_fwd_rows,
    xattn_bwd,
    xattn_bwd_workspace_size,
    xattn_fwd,
    xattn_workspace_size,
)
