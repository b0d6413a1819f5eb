"""The oracle: a plain fp64 CPU statement of the fused inference attention path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package; the product library never uses it.
The arithmetic lives in ``fia_oracle.c`` (plain C, fp64, built with
``-ffp-contract=off``); this module compiles it with gcc and marshals numpy
arrays into it.  It shares no code with the CUDA path.

Functions and the passages they follow:

* ``decode``   -- aclnnIncreFlashAttentionV3, "Function" (softmax attention with
  scaleValue) and "Constraints / page attention" (block table addressing);
  aclnnFlashAttentionScoreV4 "计算公式" (learnable sink).
* ``prefill``  -- FusedInferAttentionScore 全解析 (prefill mode, rightDownCausal);
  aclnnFlashAttentionScoreV4 "约束说明" (TND, cumulative sequence lengths).
* ``rau``      -- aclnnRingAttentionUpdate "计算公式", read with each partial
  weighted by its own softmax sum (the printed formula drops those factors).
* ``dequant_i8`` -- per-channel antiquant (x - offset) * scale in fp32.
* ``decode(mask=...)`` -- aclnnIncreFlashAttentionV3 parameter table, attenMask
  (B, 1, 1, S): nonzero bytes remove keys from the softmax.
* ``post_quant`` -- aclnnIncreFlashAttentionV3 parameter table and constraints,
  quantScale2 / quantOffset2 (int8 output, per tensor or per channel).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "fia_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None

# this interface's dtype codes (match the enum in fia_oracle.c)
F32, F16, BF16, I8, F64 = 0, 1, 2, 3, 4

GCC_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC"]


def compile_source(src: str, out: str) -> str:
    """Compile one oracle C source into a shared library (gcc, OpenMP, no FMA contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile fia_oracle.c into liboracle.so next to it, if missing or stale."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_decode.argtypes = [P, i32, P, P, i32, P, i64, P, i32, i32, i32, i32, i32, i64,
                                  dbl, P, P, P, P, i64, i64, i64, i32, P, i64, i32, P, P, P]
    lib.oracle_decode.restype = i32
    lib.oracle_prefill.argtypes = [P, P, P, i32, P, P, i32, i32, i32, i32, dbl, i32, i64, i64, P,
                                   P, i64, i32, P, P, P]
    lib.oracle_prefill.restype = i32
    lib.oracle_rau.argtypes = [P, P, P, P, P, P, i64, i32, i32, P, P, P]
    lib.oracle_rau.restype = i32
    lib.oracle_dequant_i8.argtypes = [ctypes.c_int8, ctypes.c_float, ctypes.c_float]
    lib.oracle_dequant_i8.restype = ctypes.c_float
    lib.oracle_dequant_i8_array.argtypes = [P, P, P, i64, P]
    lib.oracle_dequant_i8_array.restype = None
    lib.oracle_gather_rows.argtypes = [P, i32, P, i64, i32, i32, i64, i32, i32, i32, P]
    lib.oracle_gather_rows.restype = i32
    lib.oracle_post_quant.argtypes = [P, i64, i64, P, P, i32, P, P]
    lib.oracle_post_quant.restype = None
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i32
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _dtype_code(a: np.ndarray, declared: int | None) -> int:
    if declared is not None:
        return declared
    return {np.dtype(np.float32): F32, np.dtype(np.float64): F64, np.dtype(np.int8): I8}[a.dtype]


class Oracle:
    """numpy front end over one compiled copy of the oracle's C source."""

    def __init__(self, path: str):
        self.path = path
        self._lib = _bind(path)

    def max_threads(self) -> int:
        return self._lib.oracle_max_threads()

    def dequant_i8(self, x: int, offset: float, scale: float) -> float:
        """One fp32 antiquant step, exactly as the oracle's decode uses it."""
        return self._lib.oracle_dequant_i8(int(x), float(offset), float(scale))

    def dequant_i8_array(self, codes, offset, scale):
        """Element-wise antiquant of int8 codes with per-element fp32 offset and scale."""
        codes = np.ascontiguousarray(codes, dtype=np.int8)
        offset = np.ascontiguousarray(np.broadcast_to(offset, codes.shape), dtype=np.float32)
        scale = np.ascontiguousarray(np.broadcast_to(scale, codes.shape), dtype=np.float32)
        out = np.zeros(codes.shape, np.float32)
        self._lib.oracle_dequant_i8_array(_ptr(codes), _ptr(offset), _ptr(scale), codes.size, _ptr(out))
        return out

    def gather_rows(self, cache, block_table, b, hk, L, block_size):
        """Stored rows of tokens 0..L-1 of (b, hk) from a paged pool, as raw elements."""
        cache = np.ascontiguousarray(cache)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        _, Nkv, _, D = cache.shape
        dst = np.zeros((L, D), cache.dtype)
        rc = self._lib.oracle_gather_rows(_ptr(cache), cache.dtype.itemsize, _ptr(bt), int(bt.shape[1]), int(b),
                                          int(hk), int(L), int(Nkv), int(D), int(block_size), _ptr(dst))
        if rc != 0:
            raise ValueError("oracle_gather_rows met a negative block index")
        return dst

    def decode(self, q, k_cache, v_cache, seq_lens, *, Nq, Nkv, D, scale, q_dtype=None, kv_dtype=None,
               block_table=None, block_size=0, kv_rows=0, aq_scale=None, aq_offset=None, sink=None,
               mask=None, band=None, q_len=1, rows=None, nthreads=0):
        """Decode attention (query S = 1).

        q: (B, Nq, D) array (uint16 bits with q_dtype=F16/BF16, or float32/float64).
        k_cache, v_cache: paged (num_blocks, Nkv, block_size, D) when block_table is
        given, else contiguous (B, Nkv, kv_rows, D).  int8 caches need aq_scale
        (2, Nkv, D) float32 and optionally aq_offset.  mask: (B, S) bytes (bool,
        int8 or uint8; S >= every length), nonzero = key masked out.  band: (pre_tokens,
        next_tokens), keys L - 1 - pre .. L - 1 + next of each batch.  q_len = s > 1: q is
        (B, s, Nq, D), position i of a batch at L - s + i sees keys up to it, and rows run
        over B * s * Nq.  Returns (out, max, sum) as
        float64 arrays of shape (R, D), (R,), (R,) where R = len(rows) or B * Nq.
        """
        q = np.ascontiguousarray(q)
        k_cache = np.ascontiguousarray(k_cache)
        v_cache = np.ascontiguousarray(v_cache)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int64)
        B = int(seq_lens.shape[0])
        bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
        bt_stride = 0 if bt is None else int(bt.shape[1])
        rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        R = B * int(q_len) * Nq if rows_a is None else int(rows_a.shape[0])
        f32 = lambda a: None if a is None else np.ascontiguousarray(a, dtype=np.float32)
        aq_scale, aq_offset, sink = f32(aq_scale), f32(aq_offset), f32(sink)
        if mask is not None:
            mask = np.ascontiguousarray(np.asarray(mask).reshape(B, -1).view(np.uint8) != 0, dtype=np.uint8)
        mask_stride = 0 if mask is None else int(mask.shape[1])
        out = np.zeros((R, D), np.float64)
        mx = np.zeros(R, np.float64)
        sm = np.zeros(R, np.float64)
        rc = self._lib.oracle_decode(
            _ptr(q), _dtype_code(q, q_dtype), _ptr(k_cache), _ptr(v_cache),
            _dtype_code(k_cache, kv_dtype), _ptr(bt), bt_stride, _ptr(seq_lens),
            B, Nq, Nkv, D, block_size, kv_rows, float(scale), _ptr(aq_scale),
            _ptr(aq_offset), _ptr(sink), _ptr(mask), mask_stride,
            int(band[0]) if band is not None else 1 << 62, int(band[1]) if band is not None else 0,
            int(q_len), _ptr(rows_a), 0 if rows_a is None else R,
            nthreads, _ptr(out), _ptr(mx), _ptr(sm))
        if rc != 0:
            raise ValueError("oracle_decode rejected its arguments")
        return out, mx, sm

    def prefill(self, q, k, v, cu_q, cu_kv, *, Nq, Nkv, D, scale, causal=True, dtype=None, sink=None,
                rows=None, nthreads=0, band=None):
        """Prefill attention in TND layout.  q: (T, Nq, D); k, v: (Tkv, Nkv, D);
        cu_q / cu_kv: B + 1 cumulative lengths from 0.  band=(pre_tokens, next_tokens)
        selects sparseMode 4 (and overrides causal).  Returns (out, max, sum) in
        float64 for the rows (t * Nq + h) asked for, or for all T * Nq rows."""
        q, k, v = (np.ascontiguousarray(a) for a in (q, k, v))
        cu_q = np.ascontiguousarray(cu_q, dtype=np.int64)
        cu_kv = np.ascontiguousarray(cu_kv, dtype=np.int64)
        B = int(cu_q.shape[0]) - 1
        T = int(cu_q[-1])
        rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        R = T * Nq if rows_a is None else int(rows_a.shape[0])
        sink = None if sink is None else np.ascontiguousarray(sink, dtype=np.float32)
        out = np.zeros((R, D), np.float64)
        mx = np.zeros(R, np.float64)
        sm = np.zeros(R, np.float64)
        rc = self._lib.oracle_prefill(
            _ptr(q), _ptr(k), _ptr(v), _dtype_code(q, dtype), _ptr(cu_q), _ptr(cu_kv),
            B, Nq, Nkv, D, float(scale), 4 if band is not None else (3 if causal else 0),
            int(band[0]) if band is not None else 0, int(band[1]) if band is not None else 0, _ptr(sink), _ptr(rows_a),
            0 if rows_a is None else R, nthreads, _ptr(out), _ptr(mx), _ptr(sm))
        if rc != 0:
            raise ValueError("oracle_prefill rejected its arguments")
        return out, mx, sm

    def post_quant(self, x, scale2, offset2=None):
        """int8 output quantisation of x (rows, N, D) or (rows, C): returns (y, code), y the
        unrounded fp64 value and code the int8 result.  scale2/offset2: one value (per
        tensor) or N * D values (per channel)."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        rows = int(x.shape[0])
        C = int(x.size // max(rows, 1))
        s2 = np.ascontiguousarray(np.asarray(scale2, dtype=np.float32).reshape(-1))
        o2 = None if offset2 is None else np.ascontiguousarray(np.asarray(offset2, dtype=np.float32).reshape(-1))
        per_channel = int(s2.size != 1)
        if per_channel and s2.size != C or (o2 is not None and o2.size != s2.size):
            raise ValueError("post_quant: scale2/offset2 must hold 1 or N * D values")
        y = np.zeros(x.shape, np.float64)
        code = np.zeros(x.shape, np.int8)
        self._lib.oracle_post_quant(_ptr(x), rows, C, _ptr(s2), _ptr(o2), per_channel, _ptr(y), _ptr(code))
        return y, code

    def rau(self, prev_out, prev_max, prev_sum, cur_out, cur_max, cur_sum):
        """RingAttentionUpdate on fp64 arrays: out (rows, N, D), max/sum (rows, N)."""
        a = [np.ascontiguousarray(x, dtype=np.float64) for x in
             (prev_out, prev_max, prev_sum, cur_out, cur_max, cur_sum)]
        rows, N, D = a[0].shape
        out = np.zeros((rows, N, D), np.float64)
        mx = np.zeros((rows, N), np.float64)
        sm = np.zeros((rows, N), np.float64)
        self._lib.oracle_rau(*[_ptr(x) for x in a], rows, N, D, _ptr(out), _ptr(mx), _ptr(sm))
        return out, mx, sm


def default() -> Oracle:
    """The oracle built from fia_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def max_threads() -> int:
    return default().max_threads()


def dequant_i8(x, offset, scale):
    return default().dequant_i8(x, offset, scale)


def decode(*args, **kw):
    return default().decode(*args, **kw)


def prefill(*args, **kw):
    return default().prefill(*args, **kw)


def rau(*args, **kw):
    return default().rau(*args, **kw)


def post_quant(*args, **kw):
    return default().post_quant(*args, **kw)
