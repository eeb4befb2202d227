"""gated_delta_rule_29_gb300 -- GB300-native (sm_103a) chunked Gated DeltaNet forward.

The computation lives in liblinattn.so (C ABI: include/liblinattn.h), built
in-tree from csrc/ by ``_build.build()``.  This package is its thin Python
binding: ``gdn_fwd``, ``gdn_bwd``, ``gdn_summary``, ``gdn_summary_bwd`` and ``gdn_decode`` marshal torch tensors
into the C structs and launch on the current CUDA stream.  There is no CPU fallback.
"""
from .api import (checkpoint_rows, gdn_bwd, gdn_decode, gdn_fwd, gdn_fwd_host, gdn_summary,  # noqa: F401
                  gdn_summary_bwd, read_status, workspace_bytes)
from . import binding  # noqa: F401
from .autograd import gdn_attention  # noqa: F401

__all__ = ["gdn_fwd", "gdn_fwd_host", "gdn_summary", "gdn_summary_bwd", "gdn_decode", "gdn_bwd", "gdn_attention",
           "read_status", "checkpoint_rows", "workspace_bytes", "binding"]
