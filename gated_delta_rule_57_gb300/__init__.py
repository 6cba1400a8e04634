"""GB300-native Kimi Delta Attention (KDA): chunked prefill and decode.

The computation lives in ``libkda.so`` (hand-written sm_103a CUDA kernels
behind the C ABI of ``include/kda.h``); this package is its thin binding.
Importing the package does not load the CUDA library; the first call does.
"""
from .kda import (  # noqa: F401
    KDA_BF16, KDA_DEV_DECAY_RANGE, KDA_DEV_NONFINITE, KDA_DEV_TIMEOUT, KDA_F32, KdaError,
    kda_chunk_fwd, kda_chunk_fwd_ckpt, kda_chunk_fwd_segmented, kda_chunk_fwd_segmented_noalloc,
    kda_chunk_fwd_segment_plan, kda_chunk_fwd_segmented_workspace_size,
    kda_chunk_fwd_segments_hint, kda_chunk_fwd_slice_correct, kda_chunk_fwd_slice_transition,
    kda_chunk_fwd_workspace_size, kda_decode_multi, kda_decode_step, kda_state_scan, lib,
    status_string,
)

__all__ = ["kda_chunk_fwd", "kda_chunk_fwd_ckpt", "kda_chunk_fwd_segmented",
           "kda_chunk_fwd_segmented_noalloc",
           "kda_chunk_fwd_segmented_workspace_size", "kda_chunk_fwd_segments_hint",
           "kda_chunk_fwd_segment_plan", "kda_decode_step",
           "kda_decode_multi", "kda_chunk_fwd_workspace_size", "kda_chunk_fwd_slice_transition",
           "kda_chunk_fwd_slice_correct", "kda_state_scan", "lib", "status_string", "KdaError"]
