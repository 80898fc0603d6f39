"""GB300-native Kimi Delta Attention (KDA) chunk scan and decode step.

The compute lives in ``libkda.so`` (hand-written CUDA for sm_103a behind a C
ABI declared in ``include/kda.h``).  ``gated_delta_rule_41_gb300.kda`` is the
thin Python binding: it marshals torch tensors into the C calls and nothing
else.  The library is loaded on first use; if it is missing, every call
raises instead of falling back to another implementation.
"""
from .kda import (  # noqa: F401
    KdaError, SavedForward, chunk_kda_fwd, chunk_kda_bwd, chunk_kda_fwd_varlen,
    chunk_kda_bwd_varlen, recurrent_step, workspace_bytes,
    library_path,
    load_library, check, timing_enable, timing_read,
)
