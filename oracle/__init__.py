"""Float64 CPU oracle (test infrastructure only; see ll_oracle's header)."""
from .ll_oracle import (  # noqa: F401
    OracleCache, OracleLayer, attention_flops, block_causal_visible, frame_of_slot,
    lkv_tokens, masked_attention, resident_frames, sink_frames, slot_of_frame,
    visible_frames, window_frames,
)
