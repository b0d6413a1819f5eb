"""ctypes binding of libfia_gb300.so: argument marshalling only.

Each function here has the name of the C entry point it calls and passes torch
tensors' device addresses, shapes and the current CUDA stream through to it.
All computation happens in the library's CUDA kernels; if the library has not
been built, importing this module raises an error instead of falling back to
anything else.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfia_gb300.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "fia.h")

F32, F16, BF16, I8 = 0, 1, 2, 3
SUCCESS, ERR_PARAM_NULLPTR, ERR_PARAM_INVALID, ERR_RUNTIME, ERR_INNER_TILING = 0, 161001, 161002, 361001, 561002
STATUS_WAIT_TIMEOUT, STATUS_BAD_BLOCK_INDEX, STATUS_LENGTH_CLAMPED, STATUS_BAD_SEQLENS = 1, 2, 4, 8

_TORCH_TO_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16, torch.int8: I8}


class FiaError(RuntimeError):
    """A non-zero status from the library, with the library's own message."""

    def __init__(self, code: int, func: str, message: str):
        super().__init__(f"{func} returned {code}: {message}")
        self.code = code


class PrefillOptions(ctypes.Structure):
    """fia_prefill_options of include/fia.h."""
    _fields_ = [("pre_tokens", ctypes.c_int64), ("next_tokens", ctypes.c_int64), ("block_table", ctypes.c_void_p),
                ("bt_stride", ctypes.c_int64), ("seq_lens_kv", ctypes.c_void_p), ("block_size", ctypes.c_int),
                ("num_blocks", ctypes.c_int64), ("kv_layout", ctypes.c_int), ("quant_scale2", ctypes.c_void_p),
                ("quant_offset2", ctypes.c_void_p), ("quant2_per_channel", ctypes.c_int)]


class DecodeOptions(ctypes.Structure):
    """fia_decode_options of include/fia.h."""
    _fields_ = [("kv_layout", ctypes.c_int), ("antiquant_mode", ctypes.c_int), ("softmax_lse", ctypes.c_void_p),
                ("atten_mask", ctypes.c_void_p), ("atten_mask_stride", ctypes.c_int64),
                ("quant_scale2", ctypes.c_void_p), ("quant_offset2", ctypes.c_void_p),
                ("quant2_per_channel", ctypes.c_int), ("band", ctypes.c_int), ("pre_tokens", ctypes.c_int64),
                ("next_tokens", ctypes.c_int64), ("q_len", ctypes.c_int)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with attention_ifa_fia_gb300.build.build() "
                          "(nvcc for sm_103a); there is no other implementation to fall back to")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u32, dbl, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint,
                                 ctypes.c_double, ctypes.c_size_t)
    sig = {
        "fia_last_error": ([], ctypes.c_char_p),
        "fia_device_status": ([P, ctypes.POINTER(u32)], i32),
        "fia_decode_workspace_size": ([i32, i32, i32, i32, i32, i32, i32, ctypes.POINTER(sz)], i32),
        "fia_decode": ([P, i32, P, P, i32, P, i64, P, i32, i32, i32, i32, i32, i32, i64, dbl, P, P, P, P, P, P,
                        i32, P, sz, P], i32),
        "fia_decode_noalloc": ([P, i32, P, P, i32, P, i64, P, i32, i32, i32, i32, i32, i32, i64, dbl, P, P, P, P,
                                P, P, i32, P], i32),
        "fia_decode_ex": ([P, i32, P, P, i32, P, i64, P, i32, i32, i32, i32, i32, i32, i64, dbl, P, P, P, P, P, P,
                           i32, P, sz, P, ctypes.POINTER(DecodeOptions)], i32),
        "fia_prefill_workspace_size": ([i32, i32, i32, i32, i32, ctypes.POINTER(sz)], i32),
        "fia_prefill": ([P, P, P, i32, P, P, i32, i64, i64, i32, i32, i32, i32, i32, dbl, i32, P, P, P, P, P, sz,
                         P], i32),
        "fia_prefill_ex": ([P, P, P, i32, P, P, i32, i64, i64, i32, i32, i32, i32, i32, dbl, i32, P, P, P, P, P,
                            sz, P, ctypes.POINTER(PrefillOptions)], i32),
        "ring_attention_update": ([P, P, P, P, P, P, i32, i64, i32, i32, P, P, P, P], i32),
        "fia_debug_dequant": ([P, P, P, i64, P, P], i32),
        "fia_trace_enable": ([i32], i32),
        "fia_trace_collect": ([i32, ctypes.POINTER(dbl), ctypes.POINTER(i32)], i32),
        "fia_debug_gather": ([P, i32, P, i64, P, i32, i32, i32, i32, i32, i64, i32, i32, P, P], i32),
        "fia_debug_i8_codes": ([P, i64, P, P], i32),
        "fia_debug_i8_qprep": ([P, i32, P, P, i32, i32, i32, dbl, P, sz, P, P, P, P], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


_lib = _load()


def header_functions() -> list:
    """Names of the functions include/fia.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(\w+)\s*\(", text, flags=re.M)))


def library() -> ctypes.CDLL:
    return _lib


def _check(rc: int, func: str):
    if rc != SUCCESS:
        raise FiaError(rc, func, _lib.fia_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def dtype_code(t: torch.Tensor) -> int:
    return _TORCH_TO_CODE[t.dtype]


KERNEL_DECODE_PLAN, KERNEL_DECODE_ATTENTION, KERNEL_DECODE_MERGE, KERNEL_PREFILL, KERNEL_RAU = 0, 1, 2, 3, 4


def fia_trace_enable(on: bool = True) -> None:
    _check(_lib.fia_trace_enable(1 if on else 0), "fia_trace_enable")


def fia_trace_collect(kernel: int) -> Tuple[float, int]:
    """(summed device ms, launches) of one kernel since the last collect on this thread."""
    ms, n = ctypes.c_double(0.0), ctypes.c_int(0)
    _check(_lib.fia_trace_collect(int(kernel), ctypes.byref(ms), ctypes.byref(n)), "fia_trace_collect")
    return ms.value, n.value


def fia_device_status(stream=None) -> int:
    flags = ctypes.c_uint(0)
    _check(_lib.fia_device_status(_stream(stream), ctypes.byref(flags)), "fia_device_status")
    return flags.value


# ----------------------------------------------------------------------------- decode
KV_BNNBSD, KV_BNBSH = 0, 1            # k/v cache (num_blocks, Nkv, bs, D) or (num_blocks, bs, Nkv * D)
AQ_PER_CHANNEL, AQ_PER_TENSOR = 0, 1  # antiquant scale/offset (2, Nkv, D) or (2,)


def fia_decode_workspace_size(B: int, Nq: int, Nkv: int, D: int, max_kv_len: int, block_size: int,
                              num_splits: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.fia_decode_workspace_size(B, Nq, Nkv, D, max_kv_len, block_size, num_splits, ctypes.byref(n)),
           "fia_decode_workspace_size")
    return n.value


def fia_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
               actual_seq_lengths: torch.Tensor, *, max_kv_len: int, num_heads: int, num_kv_heads: int = 0,
               scale: Optional[float] = None, antiquant_scale=None, antiquant_offset=None, sink=None,
               out: Optional[torch.Tensor] = None, softmax_max: Optional[torch.Tensor] = None,
               softmax_sum: Optional[torch.Tensor] = None, num_splits: int = 0,
               workspace: Optional[torch.Tensor] = None, stream=None, kv_layout: int = KV_BNNBSD,
               antiquant_mode: int = AQ_PER_CHANNEL, softmax_lse: Optional[torch.Tensor] = None,
               atten_mask: Optional[torch.Tensor] = None, quant_scale2: Optional[torch.Tensor] = None,
               quant_offset2: Optional[torch.Tensor] = None, pre_tokens: Optional[int] = None,
               next_tokens: Optional[int] = None, q_len: int = 1,
               _force_ex: bool = False) -> Tuple[torch.Tensor, Optional[torch.Tensor], Optional[torch.Tensor]]:
    """Paged decode attention.  q: (B, Nq, D) (any layout of that memory); k/v_cache:
    (num_blocks, Nkv, block_size, D), or with kv_layout=KV_BNBSH (num_blocks, block_size,
    Nkv * D); block_table int32 (B, width); actual_seq_lengths int64 (B,) on the device.
    antiquant_mode=AQ_PER_TENSOR takes scale/offset of shape (2,); softmax_lse (B, Nq)
    receives max + ln(sum).  atten_mask: (B, S) / (B, 1, S) / (B, 1, 1, S) bool, int8 or
    uint8, 1 = key masked out, S >= max_kv_len.  quant_scale2 (and quant_offset2): fp32 of
    1 or Nq * D values; out is then int8.  pre_tokens / next_tokens: the band around the
    query (keys L - 1 - pre .. L - 1 + next).  q_len = s > 1: q is (B, s, Nq, D), s query
    positions per batch, position i at key L - s + i seeing keys up to it; out (B, s, Nq, D)
    and max / sum / lse (B, s, Nq).  Returns (out, softmax_max, softmax_sum)."""
    B, D = int(q.shape[0]), int(q.shape[-1])
    num_blocks = int(k_cache.shape[0])
    block_size = int(k_cache.shape[1] if kv_layout == KV_BNBSH else k_cache.shape[2])
    nkv = num_kv_heads if num_kv_heads else num_heads
    if scale is None:
        scale = D ** -0.5
    out_dtype = torch.int8 if quant_scale2 is not None else q.dtype
    if out is None:
        shape = (B, num_heads, D) if q_len <= 1 else (B, q_len, num_heads, D)
        out = torch.empty(shape, dtype=out_dtype, device=q.device)
    elif out.dtype != out_dtype and quant_offset2 is None:  # (an offset alone is the library's error)
        raise ValueError(f"out must be {out_dtype} (got {out.dtype})")
    mask_stride = 0
    if atten_mask is not None:
        if atten_mask.dtype not in (torch.bool, torch.int8, torch.uint8) or not atten_mask.is_contiguous():
            raise ValueError("atten_mask must be a contiguous bool, int8 or uint8 tensor")
        mask_stride = int(atten_mask.shape[-1])
        if atten_mask.numel() != B * mask_stride:
            raise ValueError("atten_mask must have shape (B, S), (B, 1, S) or (B, 1, 1, S)")
    q2_per_channel = 0
    if quant_scale2 is not None:
        n2 = quant_scale2.numel()
        if n2 not in (1, num_heads * D) or quant_scale2.dtype != torch.float32:
            raise ValueError("quant_scale2 must be fp32 with 1 or Nq * D values")
        if quant_offset2 is not None and (quant_offset2.numel() != n2 or quant_offset2.dtype != torch.float32):
            raise ValueError("quant_offset2 must match quant_scale2")
        q2_per_channel = int(n2 != 1)
    if workspace is None:
        nbytes = fia_decode_workspace_size(B, num_heads * max(q_len, 1), nkv, D, max_kv_len, block_size, num_splits)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    args = (_ptr(q), dtype_code(q), _ptr(k_cache), _ptr(v_cache), dtype_code(k_cache), _ptr(block_table),
            int(block_table.shape[1]), _ptr(actual_seq_lengths), int(max_kv_len), B, num_heads, nkv, D, block_size,
            num_blocks, float(scale), _ptr(antiquant_scale), _ptr(antiquant_offset), _ptr(sink), _ptr(out),
            _ptr(softmax_max), _ptr(softmax_sum), int(num_splits), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(stream))
    band = pre_tokens is not None or next_tokens is not None
    plain = (kv_layout == KV_BNNBSD and antiquant_mode == AQ_PER_CHANNEL and softmax_lse is None
             and atten_mask is None and quant_scale2 is None and quant_offset2 is None and not band
             and q_len <= 1)
    if plain and not _force_ex:
        _check(_lib.fia_decode(*args), "fia_decode")
    else:
        opts = DecodeOptions(int(kv_layout), int(antiquant_mode), _ptr(softmax_lse), _ptr(atten_mask), mask_stride,
                             _ptr(quant_scale2), _ptr(quant_offset2), q2_per_channel, int(band),
                             int(pre_tokens if pre_tokens is not None else 1 << 40),
                             int(next_tokens if next_tokens is not None else 1 << 40), int(q_len))
        _check(_lib.fia_decode_ex(*args, ctypes.byref(opts)), "fia_decode_ex")
    return out, softmax_max, softmax_sum


def fia_decode_ex(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                  actual_seq_lengths: torch.Tensor, *, kv_layout: int = KV_BNNBSD, antiquant_mode: int = AQ_PER_CHANNEL,
                  softmax_lse: Optional[torch.Tensor] = None, atten_mask: Optional[torch.Tensor] = None,
                  quant_scale2: Optional[torch.Tensor] = None, quant_offset2: Optional[torch.Tensor] = None,
                  pre_tokens: Optional[int] = None, next_tokens: Optional[int] = None, **kw):
    """fia_decode_ex: fia_decode with the decode options (KV layout, antiquant mode,
    log-sum-exp output, attenMask, int8 post-quant output); other arguments as for
    fia_decode.  Always calls the C fia_decode_ex entry point."""
    return fia_decode(q, k_cache, v_cache, block_table, actual_seq_lengths, kv_layout=kv_layout,
                      antiquant_mode=antiquant_mode, softmax_lse=softmax_lse, atten_mask=atten_mask,
                      quant_scale2=quant_scale2, quant_offset2=quant_offset2, pre_tokens=pre_tokens,
                      next_tokens=next_tokens, _force_ex=True, **kw)


def fia_decode_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                       actual_seq_lengths: torch.Tensor, *, max_kv_len: int, num_heads: int, num_kv_heads: int = 0,
                       scale: Optional[float] = None, antiquant_scale=None, antiquant_offset=None, sink=None,
                       out: Optional[torch.Tensor] = None, softmax_max: Optional[torch.Tensor] = None,
                       softmax_sum: Optional[torch.Tensor] = None, num_splits: int = 0, stream=None):
    """fia_decode without a workspace argument: the library uses its own fixed device scratch
    (for callers that cannot allocate; see include/fia.h).  `out` must be given by callers
    that may not allocate; when omitted it is created here for convenience."""
    B, D = int(q.shape[0]), int(q.shape[-1])
    num_blocks, block_size = int(k_cache.shape[0]), int(k_cache.shape[2])
    nkv = num_kv_heads if num_kv_heads else num_heads
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty((B, num_heads, D), dtype=q.dtype, device=q.device)
    rc = _lib.fia_decode_noalloc(_ptr(q), dtype_code(q), _ptr(k_cache), _ptr(v_cache), dtype_code(k_cache),
                                 _ptr(block_table), int(block_table.shape[1]), _ptr(actual_seq_lengths),
                                 int(max_kv_len), B, num_heads, nkv, D, block_size, num_blocks, float(scale),
                                 _ptr(antiquant_scale), _ptr(antiquant_offset), _ptr(sink), _ptr(out),
                                 _ptr(softmax_max), _ptr(softmax_sum), int(num_splits), _stream(stream))
    _check(rc, "fia_decode_noalloc")
    return out, softmax_max, softmax_sum


# ----------------------------------------------------------------------------- prefill
def fia_prefill_workspace_size(B: int, Nq: int, Nkv: int, D: int, max_seqlen_q: int) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.fia_prefill_workspace_size(B, Nq, Nkv, D, max_seqlen_q, ctypes.byref(n)),
           "fia_prefill_workspace_size")
    return n.value


def fia_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                cu_seqlens_kv: torch.Tensor, *, max_seqlen_q: int, max_seqlen_kv: int, num_heads: int,
                num_kv_heads: int = 0, scale: Optional[float] = None, mask: int = 3, sink=None,
                out: Optional[torch.Tensor] = None, softmax_max=None, softmax_sum=None,
                workspace: Optional[torch.Tensor] = None, stream=None, pre_tokens: Optional[int] = None,
                next_tokens: Optional[int] = None, block_table: Optional[torch.Tensor] = None,
                seq_lens_kv: Optional[torch.Tensor] = None, kv_layout: int = KV_BNNBSD,
                quant_scale2: Optional[torch.Tensor] = None, quant_offset2: Optional[torch.Tensor] = None):
    """Prefill attention, TND.  q: (T, Nq, D); k, v: (Tkv, Nkv, D); cu_seqlens int64 (B + 1,)
    on the device.  mask 3 = rightDownCausal, 0 = none, 4 = band (pre_tokens, next_tokens
    around the rightDownCausal diagonal, through fia_prefill_ex).  With block_table (int32
    (B, width)) and seq_lens_kv (int64 (B,)), k and v are paged pools (num_blocks, Nkv,
    block_size, D), or with kv_layout=KV_BNBSH (num_blocks, block_size, Nkv * D), and
    cu_seqlens_kv may be None.  quant_scale2 (and quant_offset2): fp32 of 1 or Nq * D values;
    out is then int8.  Returns (out, softmax_max, softmax_sum)."""
    T, D = int(q.shape[0]), int(q.shape[-1])
    paged = block_table is not None
    Tkv = 0 if paged else int(k.shape[0])
    B = int(cu_seqlens_q.shape[0]) - 1
    nkv = num_kv_heads if num_kv_heads else num_heads
    if scale is None:
        scale = D ** -0.5
    out_dtype = torch.int8 if quant_scale2 is not None else q.dtype
    if out is None:
        out = torch.empty((T, num_heads, D), dtype=out_dtype, device=q.device)
    elif out.dtype != out_dtype and quant_offset2 is None:  # (an offset alone is the library's error)
        raise ValueError(f"out must be {out_dtype} (got {out.dtype})")
    q2_per_channel = 0
    if quant_scale2 is not None:
        n2 = quant_scale2.numel()
        if n2 not in (1, num_heads * D) or quant_scale2.dtype != torch.float32:
            raise ValueError("quant_scale2 must be fp32 with 1 or Nq * D values")
        if quant_offset2 is not None and (quant_offset2.numel() != n2 or quant_offset2.dtype != torch.float32):
            raise ValueError("quant_offset2 must match quant_scale2")
        q2_per_channel = int(n2 != 1)
    if workspace is None:
        nbytes = fia_prefill_workspace_size(B, num_heads, nkv, D, max_seqlen_q)
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    args = (_ptr(q), _ptr(k), _ptr(v), dtype_code(q), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), B, T, Tkv,
            int(max_seqlen_q), int(max_seqlen_kv), num_heads, nkv, D, float(scale), int(mask), _ptr(sink), _ptr(out),
            _ptr(softmax_max), _ptr(softmax_sum), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream))
    if pre_tokens is None and next_tokens is None and not paged and quant_scale2 is None and quant_offset2 is None:
        _check(_lib.fia_prefill(*args), "fia_prefill")
    else:
        bs = (int(k.shape[1]) if kv_layout == KV_BNBSH else int(k.shape[2])) if paged else 0
        opts = PrefillOptions(int(pre_tokens if pre_tokens is not None else 1 << 40),
                              int(next_tokens if next_tokens is not None else 1 << 40),
                              _ptr(block_table), int(block_table.shape[1]) if paged else 0, _ptr(seq_lens_kv), bs,
                              int(k.shape[0]) if paged else 0, int(kv_layout), _ptr(quant_scale2),
                              _ptr(quant_offset2), q2_per_channel)
        _check(_lib.fia_prefill_ex(*args, ctypes.byref(opts)), "fia_prefill_ex")
    return out, softmax_max, softmax_sum


# ----------------------------------------------------------------------------- RAU
def ring_attention_update(prev_out, prev_max, prev_sum, cur_out, cur_max, cur_sum, *, out=None, max_out=None,
                          sum_out=None, stream=None):
    """Merge two partials.  *_out: (rows, N, D) f32/f16/bf16; *_max/*_sum: (rows, N) fp32.
    Outputs default to new tensors; passing the prev_* tensors merges in place."""
    rows, N, D = (int(x) for x in prev_out.shape)
    out = torch.empty_like(prev_out) if out is None else out
    max_out = torch.empty_like(prev_max) if max_out is None else max_out
    sum_out = torch.empty_like(prev_sum) if sum_out is None else sum_out
    rc = _lib.ring_attention_update(_ptr(prev_out), _ptr(prev_max), _ptr(prev_sum), _ptr(cur_out), _ptr(cur_max),
                                    _ptr(cur_sum), dtype_code(prev_out), rows, N, D, _ptr(out), _ptr(max_out),
                                    _ptr(sum_out), _stream(stream))
    _check(rc, "ring_attention_update")
    return out, max_out, sum_out


# ----------------------------------------------------------------------------- probes
def fia_debug_dequant(codes: torch.Tensor, scale: torch.Tensor, offset: torch.Tensor, stream=None) -> torch.Tensor:
    out = torch.empty(codes.shape, dtype=torch.float32, device=codes.device)
    _check(_lib.fia_debug_dequant(_ptr(codes), _ptr(scale), _ptr(offset), codes.numel(), _ptr(out),
                                  _stream(stream)), "fia_debug_dequant")
    return out


def fia_debug_gather(k_cache: torch.Tensor, block_table: torch.Tensor, actual_seq_lengths: torch.Tensor, *,
                     max_kv_len: int, b: int, hkv: int, length: int, stream=None) -> torch.Tensor:
    num_blocks, nkv, block_size, D = (int(x) for x in k_cache.shape)
    B = int(block_table.shape[0])
    dst = torch.zeros((length, D), dtype=k_cache.dtype, device=k_cache.device)
    _check(_lib.fia_debug_gather(_ptr(k_cache), dtype_code(k_cache), _ptr(block_table), int(block_table.shape[1]),
                                 _ptr(actual_seq_lengths), int(max_kv_len), B, nkv, D, block_size, num_blocks, b,
                                 hkv, _ptr(dst), _stream(stream)), "fia_debug_gather")
    return dst


I8_QPREP_BLOCK_BYTES = 8320  # one (b, kv head) block of the int8 tensor-core query operand


def fia_debug_i8_codes(codes: torch.Tensor, stream=None) -> torch.Tensor:
    """The int8 tensor-core kernel's code -> binary16 conversion; returns int16 bit patterns."""
    out = torch.empty(codes.shape, dtype=torch.int16, device=codes.device)
    _check(_lib.fia_debug_i8_codes(_ptr(codes), codes.numel(), _ptr(out), _stream(stream)), "fia_debug_i8_codes")
    return out


def fia_debug_i8_qprep(q: torch.Tensor, antiquant_scale: torch.Tensor, antiquant_offset=None, *, num_heads: int,
                       num_kv_heads: int, scale: Optional[float] = None, stream=None):
    """The query operand of the int8 tensor-core kernel: (hi, lo) int16 bit patterns of
    shape (B, Nkv, 16, 128) and {kq, nq} fp32 of shape (B, Nkv, 16, 2)."""
    B, D = int(q.shape[0]), int(q.shape[-1])
    if scale is None:
        scale = D ** -0.5
    nblk = B * num_kv_heads
    blocks = torch.empty(max(nblk, 1) * I8_QPREP_BLOCK_BYTES, dtype=torch.uint8, device=q.device)
    hi = torch.empty((B, num_kv_heads, 16, 128), dtype=torch.int16, device=q.device)
    lo = torch.empty_like(hi)
    kn = torch.empty((B, num_kv_heads, 16, 2), dtype=torch.float32, device=q.device)
    _check(_lib.fia_debug_i8_qprep(_ptr(q), dtype_code(q), _ptr(antiquant_scale), _ptr(antiquant_offset), B,
                                   num_heads, num_kv_heads, float(scale), _ptr(blocks), blocks.numel(), _ptr(hi),
                                   _ptr(lo), _ptr(kn), _stream(stream)), "fia_debug_i8_qprep")
    return hi, lo, kn
