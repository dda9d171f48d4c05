"""fp64 CPU oracle for the Gated DeltaNet recurrence -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and has
no fallback to it.  It shares no code with the CUDA path; both sides receive
the same inputs from the seeded generators in
``invariant_linear_attention_gb300.inputs``, which hold no arithmetic of the
method.

Parity status of each function (what pins it is in ``tests/test_oracle_pins.py``):

* ``gdn_fwd``          -- pinned: identity, delta-rule projection, full forget,
                          associative recall, Kronecker brute force, split
                          invariance, linearity, GQA map, WY agreement.
* ``gdn_fwd_chunked``  -- pinned by agreement with ``gdn_fwd`` (and exactly
                          equal in exact arithmetic to it for chunk size 1).
* ``gdn_bwd``          -- pinned by central finite differences of ``gdn_fwd``
                          on every input, plus the beta=0 and one-token cases.
* ``gdn_replay_state`` -- pinned: the state rebuilt from the cache equals
                          ``gdn_fwd``'s final state; its d rows equal the
                          chunked WY form's U rows.
* ``layer_ops``        -- gates, causal conv, gated RMSNorm: pinned in
                          ``tests/test_oracle_layer_pins.py``.
"""
from .oracle import gdn_fwd, gdn_bwd, gdn_fwd_chunked, gdn_replay_state, max_threads  # noqa: F401
