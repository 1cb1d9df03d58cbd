"""kkt_solve for GB300: the chunk-local UT transform of Gated DeltaNet prefill.

    from gdn_chunkwise_ut_gb300 import kkt_solve_fwd
    T, W, U = kkt_solve_fwd(k, v, beta, C=64)            # k, v bf16 [B,T,H,128] on cuda
    o, S = gdn_chunk_state_fwd(q, k, W, U, C=64)         # the chunk recurrence that consumes W, U

The computation runs in libkkt.so (hand-written CUDA for sm_103a, C ABI in
include/kkt.h); this package only marshals torch tensors.
"""
from .api import (  # noqa: F401
    HostRunner,
    chunk_gated_delta_rule,
    device_status,
    gdn_chunk_state_fwd,
    host_workspace_bytes,
    kkt_solve_fwd,
    kkt_solve_fwd_host,
    select_kernel,
)
from ._lib import KktError  # noqa: F401

__all__ = ["kkt_solve_fwd", "kkt_solve_fwd_host", "host_workspace_bytes", "gdn_chunk_state_fwd",
           "chunk_gated_delta_rule", "device_status", "select_kernel", "HostRunner", "KktError"]
