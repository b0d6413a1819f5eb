"""Helpers for the GPU parity tests: move seeded inputs to the device, call the
library through its C interface, and compare with the oracle.

Tolerances (elementwise |gpu - oracle| <= atol + rtol * |oracle|):
  out   bf16: atol = rtol = 1e-2;  fp16: atol = rtol = 2e-3;  fp32 (RAU): 1e-5
  max, sum: rtol = 1e-4 (relative only, as stated for the fp32 softmax max and sum).
  A softmax maximum close to zero can miss a purely relative bound although the
  score behind it is as accurate as any other: a dot product of D <= 128 fp32
  products of O(1) terms carries an absolute error near 1e-7, whatever its value.
  Such rows -- |max| < 0.1 with an absolute error <= 1e-5 -- are accepted and
  recorded (NEAR_ZERO_MAX_ROWS, printed at the end of the session), so that the
  rows that need more than the relative bound are listed, not hidden.
Integer and byte results (gathered rows, dequantised codes) must be identical.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import fia_workloads as W
import oracle as OR
from fia_workloads import DeviceDecode, DevicePrefill  # noqa: F401  (re-exported for the tests)

OUT_TOL = {W.BF16: (1e-2, 1e-2), W.FP16: (2e-3, 2e-3), "fp32": (1e-5, 1e-5)}
MAX_RTOL = 1e-4
SUM_TOL = (0.0, 1e-4)
NEAR_ZERO_MAX = 0.1          # |max| below which the absolute term below may be used
NEAR_ZERO_MAX_ATOL = 1e-5
NEAR_ZERO_MAX_ROWS = []      # (test, quantity, flat index, |oracle|, abs error)


def dev_bits(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """uint16 storage bits -> device tensor of the storage dtype (bit-exact)."""
    return W.device_bits(bits, dtype, device)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(name, got, ref, atol, rtol):
    """Elementwise bound with -inf == -inf; returns (max abs err, max rel err)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    both_inf = np.isinf(got) & np.isinf(ref) & (np.sign(got) == np.sign(ref))
    g = np.where(both_inf, 0.0, got)
    r = np.where(both_inf, 0.0, ref)
    err = np.abs(g - r)
    bad = ~(err <= atol + rtol * np.abs(r))
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} outside atol={atol} rtol={rtol}; "
                             f"first at {tuple(i)}: gpu={got[tuple(i)]!r} oracle={ref[tuple(i)]!r}; "
                             f"max abs err {float(err.max()):.3g}")
    rel = err / np.maximum(np.abs(r), 1e-30)
    return float(err.max()) if err.size else 0.0, float(rel.max()) if rel.size else 0.0


def assert_close_max(name, got, ref, rtol=MAX_RTOL):
    """The softmax max (or log-sum-exp) within rtol; a row near zero (|ref| < NEAR_ZERO_MAX)
    may instead be within NEAR_ZERO_MAX_ATOL, and every such row is recorded."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    both_inf = np.isinf(got) & np.isinf(ref) & (np.sign(got) == np.sign(ref))
    g = np.where(both_inf, 0.0, got)
    r = np.where(both_inf, 0.0, ref)
    err = np.abs(g - r)
    rel_ok = err <= rtol * np.abs(r)
    near = ~rel_ok & (np.abs(r) < NEAR_ZERO_MAX) & (err <= NEAR_ZERO_MAX_ATOL)
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    for i in np.argwhere(near.reshape(-1)).reshape(-1):
        NEAR_ZERO_MAX_ROWS.append((test, name, int(i), float(abs(r.reshape(-1)[i])), float(err.reshape(-1)[i])))
    bad = ~(rel_ok | near)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{name}: {int(bad.sum())} of {bad.size} outside rtol={rtol}; first at {tuple(i)}: "
                             f"gpu={got[tuple(i)]!r} oracle={ref[tuple(i)]!r}; max abs err {float(err.max()):.3g}")
    rel = err / np.maximum(np.abs(r), 1e-30)
    return float(err.max()) if err.size else 0.0, float(rel.max()) if rel.size else 0.0


# ----------------------------------------------------------------------------- decode
def check_codes(code, y, out_ref, s_c, atol, rtol):
    """code (rows, C) int8 against the oracle's unrounded y = out_ref * s + o: the kernel
    quantises its own fp32 output, which is within (atol + rtol |out|) of out_ref, so its
    code lies within 0.5 + s (atol + rtol |out_ref|) of y after saturation."""
    c = code.astype(np.float64)
    margin = np.abs(s_c) * (atol + rtol * np.abs(out_ref))
    lo = np.clip(np.rint(y - margin), -128, 127)
    hi = np.clip(np.rint(y + margin), -128, 127)
    bad = (c < lo) | (c > hi)
    assert not bad.any(), f"{bad.sum()} codes outside the tolerance band, e.g. {np.argwhere(bad)[:4].tolist()}"


def run_decode(F, dd: DeviceDecode, num_splits=0, sink="case", max_kv_len=None, lens=None, bt=None):
    c = dd.case
    B, Nq = c.B, c.Nq
    mx = torch.full((B, Nq), float("nan"), dtype=torch.float32, device=dd.q.device)
    sm = torch.full((B, Nq), float("nan"), dtype=torch.float32, device=dd.q.device)
    out, mx, sm = F.fia_decode(dd.q, dd.k, dd.v, dd.bt if bt is None else bt, dd.lens if lens is None else lens,
                               max_kv_len=c.max_len if max_kv_len is None else max_kv_len, num_heads=Nq,
                               num_kv_heads=c.Nkv, scale=c.scale, antiquant_scale=dd.aq_scale,
                               antiquant_offset=dd.aq_offset, sink=dd.sink if sink == "case" else sink,
                               softmax_max=mx, softmax_sum=sm, num_splits=num_splits)
    return out, mx, sm


def oracle_decode(case: W.DecodeCase, rows=None, nthreads=0, sink="case", mask=None, band=None):
    code = {W.BF16: OR.BF16, W.FP16: OR.F16}
    kvc = OR.I8 if case.kv_dtype == W.INT8 else code[case.kv_dtype]
    return OR.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=case.Nq, Nkv=case.Nkv, D=case.D,
                     scale=case.scale, q_dtype=code[case.dtype], kv_dtype=kvc, block_table=case.block_table,
                     block_size=case.block_size, aq_scale=case.aq_scale, aq_offset=case.aq_offset,
                     sink=case.sink if sink == "case" else sink, mask=mask, band=band, rows=rows, nthreads=nthreads)


def compare_decode(case: W.DecodeCase, out, mx, sm, rows=None, ref=None):
    """Compare device results (full tensors) with the oracle on `rows` (b * Nq + h) or all."""
    if ref is None:
        ref = oracle_decode(case, rows=rows)
    o_ref, m_ref, s_ref = ref
    o = to_f64(out).reshape(case.B * case.Nq, case.D)
    m = to_f64(mx).reshape(-1)
    s = to_f64(sm).reshape(-1)
    if rows is not None:
        o, m, s = o[rows], m[rows], s[rows]
    atol, rtol = OUT_TOL[case.dtype]
    e_out = assert_close("out", o, o_ref, atol, rtol)
    e_max = assert_close_max("softmax_max", m, m_ref)
    e_sum = assert_close("softmax_sum", s, s_ref, *SUM_TOL)
    return {"out": e_out, "max": e_max, "sum": e_sum}


def sample_rows(case: W.DecodeCase, n: int, seed: int = 0) -> np.ndarray:
    """n random (b * Nq + h) rows plus every head of the shortest and the longest sequence."""
    rng = np.random.default_rng(seed)
    total = case.B * case.Nq
    picks = set(rng.choice(total, size=min(n, total), replace=False).tolist())
    for b in (int(np.argmin(case.lengths)), int(np.argmax(case.lengths))):
        picks.update(range(b * case.Nq, (b + 1) * case.Nq))
    return np.array(sorted(picks), np.int64)


# ----------------------------------------------------------------------------- prefill
def run_prefill(F, dp: DevicePrefill, causal=True, sink="case", band=None):
    c = dp.case
    mx = torch.full((c.T, c.Nq), float("nan"), dtype=torch.float32, device=dp.q.device)
    sm = torch.full((c.T, c.Nq), float("nan"), dtype=torch.float32, device=dp.q.device)
    return F.fia_prefill(dp.q, dp.k, dp.v, dp.cu_q, dp.cu_kv, max_seqlen_q=int(c.lengths_q.max(initial=0)),
                         max_seqlen_kv=int(c.lengths_kv.max(initial=0)), num_heads=c.Nq, num_kv_heads=c.Nkv,
                         scale=c.scale, mask=4 if band is not None else (3 if causal else 0),
                         sink=dp.sink if sink == "case" else sink, softmax_max=mx, softmax_sum=sm,
                         pre_tokens=None if band is None else band[0], next_tokens=None if band is None else band[1])


def oracle_prefill(case: W.PrefillCase, rows=None, causal=True, sink="case", nthreads=0, band=None):
    code = {W.BF16: OR.BF16, W.FP16: OR.F16}[case.dtype]
    return OR.prefill(case.q, case.k, case.v, case.cu_q, case.cu_kv, Nq=case.Nq, Nkv=case.Nkv, D=case.D,
                      scale=case.scale, causal=causal, dtype=code, sink=case.sink if sink == "case" else sink,
                      rows=rows, nthreads=nthreads, band=band)


def compare_prefill(case: W.PrefillCase, out, mx, sm, rows=None, ref=None, causal=True, band=None):
    if ref is None:
        ref = oracle_prefill(case, rows=rows, causal=causal, band=band)
    o = to_f64(out).reshape(case.T * case.Nq, case.D)
    m = to_f64(mx).reshape(-1)
    s = to_f64(sm).reshape(-1)
    if rows is not None:
        o, m, s = o[rows], m[rows], s[rows]
    atol, rtol = OUT_TOL[case.dtype]
    return {"out": assert_close("out", o, ref[0], atol, rtol),
            "max": assert_close_max("softmax_max", m, ref[1]),
            "sum": assert_close("softmax_sum", s, ref[2], *SUM_TOL)}


def sample_prefill_rows(case: W.PrefillCase, n: int, seed: int = 0) -> np.ndarray:
    """n random (t * Nq + h) rows plus all heads of the first and last token of every sequence."""
    rng = np.random.default_rng(seed)
    total = case.T * case.Nq
    picks = set(rng.choice(total, size=min(n, total), replace=False).tolist())
    for b in range(case.B):
        for t in {int(case.cu_q[b]), int(case.cu_q[b + 1]) - 1}:
            if case.cu_q[b] <= t < case.cu_q[b + 1]:
                picks.update(range(t * case.Nq, (t + 1) * case.Nq))
    return np.array(sorted(picks), np.int64)
