"""ExpCast FP8 attention for GB300 (sm_103a).

The computation lives in libovc (CUDA, C ABI in include/ovc.h); this package
is its Python binding.  ``attention(q, k, v)`` is the full call.  Importing
the package does not load the library; the first call does, and fails loudly
if it has not been built.
"""
from .api import (CapturedAttention, OvcError, Prepared, Repair, attention, attention_prepared, attention_probe,
                  attention_v_repair, attention_workspace_bytes, attn_flags, group_v, device_status, flops, prepare, prepare_v_repair,
                  prepare_workspace_bytes, repair_workspace_bytes, baseline_attention)

__all__ = ["CapturedAttention", "OvcError", "Prepared", "Repair", "attention", "attention_prepared", "attention_probe",
           "attention_v_repair", "attention_workspace_bytes", "attn_flags", "group_v", "device_status", "flops", "prepare", "prepare_v_repair",
           "prepare_workspace_bytes", "repair_workspace_bytes", "baseline_attention"]
