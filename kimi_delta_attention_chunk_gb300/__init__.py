"""GB300-native Kimi Delta Attention (KDA) forward.

The compute lives in ``libkda.so`` (CUDA for sm_103a behind the C ABI declared
in ``include/kda.h``); :mod:`.kda` is a thin ctypes binding that marshals
torch tensors and the current stream into those calls; :mod:`.cp` builds
context-parallel prefill (a sequence split into segments, across ranks or on
one device) from those calls.  Importing the package does not load the
library; the first call does, and fails loudly if the library is missing.
"""
from .kda import (  # noqa: F401
    KDAError,
    SIGNATURES,
    bwd_workspace_size,
    check_range,
    chunk_bwd,
    chunk_fwd,
    chunk_fwd_fused,
    chunk_fwd_noalloc,
    gate_proj,
    gate_proj_workspace_size,
    inject_wait_timeout,
    library_path,
    load_library,
    output_gate,
    recurrent_step,
    set_wait_limit,
    state_compose,
    trace_events,
    workspace_size,
)
