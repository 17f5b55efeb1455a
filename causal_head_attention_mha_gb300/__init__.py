"""Fused causal multi-head attention for GB300 (sm_103a).

The computation lives in ``lib/libmha.so`` (hand-written CUDA behind a C
ABI, see ``include/mha.h``); :mod:`.binding` marshals torch tensors to it.
"""
from .binding import (MHAError, mha_decode, mha_decode_ex, mha_decode_f16, mha_decode_noalloc, mha_decode_num_splits, mha_fwd,
                      mha_fwd_ex, mha_fwd_f16, mha_fwd_f32, mha_fwd_varlen, mha_fwd_varlen_f16, mha_get_device_status, mha_out_proj, mha_prefill_schedule, mha_prefill_wide_schedule, mha_qkv_proj, mha_set_fault_injection,
                      mha_set_wait_limit_ns, mha_status_string, library_path, load_library)

__all__ = ["MHAError", "mha_fwd", "mha_fwd_ex", "mha_fwd_f16", "mha_fwd_f32", "mha_fwd_varlen", "mha_fwd_varlen_f16", "mha_decode", "mha_decode_ex", "mha_decode_f16",
           "mha_decode_noalloc", "mha_decode_num_splits", "mha_get_device_status", "mha_out_proj", "mha_prefill_schedule", "mha_prefill_wide_schedule", "mha_qkv_proj", "mha_set_fault_injection",
           "mha_set_wait_limit_ns", "mha_status_string", "library_path", "load_library"]
