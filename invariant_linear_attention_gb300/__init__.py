"""Batch-invariant Gated DeltaNet kernels for GB300 (sm_103a).

One recurrent kernel serves prefill, decode and the trainer forward with
bit-identical results per sequence (whatever shares the batch, however the
tokens arrive); a chunked WY-form backward supplies gradients.  The compute
lives in libgdn.so (C ABI: include/gdn.h for the recurrence,
include/gdn_layer.h for the gate activations, the short causal conv with its
state cache, and the gated RMSNorm around it, include/gdn_replay.h for the
chunk-order-replaying variant); this package is its ctypes
binding plus the seeded synthetic-input generators.
"""
from .binding import (  # noqa: F401
    ConvShape,
    GdnError,
    GdnShape,
    gdn_causal_conv1d_fwd,
    gdn_causal_conv1d_update,
    gdn_gated_rmsnorm,
    gdn_gates,
    gdn_chunk_bwd,
    gdn_decode_step,
    gdn_recurrent_fwd,
    gdn_recurrent_fwd_noalloc,
    gdn_recurrent_fwd_snapshots,
    gdn_replay_decode,
    gdn_replay_prefill,
    gdn_workspace_size,
    lib,
    make_shape,
    read_device_error,
    replay_block_floats,
    replay_state_new,
    replay_views,
    snapshot_offsets,
    status_string,
)
