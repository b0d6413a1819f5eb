"""attention_ifa_fia_gb300: fused inference attention for one GB300 (sm_103a).

The compute lives in libfia_gb300.so (hand-written CUDA; C interface in
include/fia.h).  This package is its Python binding: the functions below carry
the C entry points' names and only marshal torch tensors into them.
"""
from ._binding import (AQ_PER_CHANNEL, AQ_PER_TENSOR, BF16, F16, F32, I8, KERNEL_DECODE_ATTENTION,
                       KERNEL_DECODE_MERGE, KERNEL_DECODE_PLAN, KERNEL_PREFILL, KERNEL_RAU, KV_BNBSH, KV_BNNBSD,
                       FiaError, fia_debug_dequant, fia_debug_gather, fia_debug_i8_codes, fia_debug_i8_qprep,
                       fia_decode, fia_decode_ex, fia_decode_noalloc, fia_decode_workspace_size, fia_device_status,
                       fia_prefill, fia_prefill_workspace_size, fia_trace_collect, fia_trace_enable,
                       header_functions, library, ring_attention_update)

__all__ = ["FiaError", "fia_decode", "fia_decode_ex", "fia_decode_noalloc", "fia_decode_workspace_size",
           "fia_prefill", "fia_prefill_workspace_size", "ring_attention_update", "fia_device_status",
           "fia_debug_dequant", "fia_debug_gather", "fia_debug_i8_codes", "fia_debug_i8_qprep",
           "fia_trace_enable", "fia_trace_collect", "header_functions", "library", "F32", "F16", "BF16", "I8",
           "KERNEL_DECODE_PLAN", "KERNEL_DECODE_ATTENTION", "KERNEL_DECODE_MERGE", "KERNEL_PREFILL", "KERNEL_RAU",
           "KV_BNNBSD", "KV_BNBSH", "AQ_PER_CHANNEL", "AQ_PER_TENSOR"]
