"""GPU parity of the decode variants of fia_decode_ex against the oracle.

aclnnIncreFlashAttentionV3, "Constraints / page attention": besides (blocknum, KV_N,
blocksize, D), the paged cache may be laid out (blocknum, blocksize, H), H = KV_N * D;
"antiquantScale / antiquantOffset": a per-tensor form of shape (2).
FusedInferAttentionScore: the softmaxLse output, ln of the softmax denominator.
aclnnIncreFlashAttentionV3 parameter table: attenMask (B, 1, 1, S), 1 = key masked out;
quantScale2 / quantOffset2, an int8 output quantised per tensor or per channel.

The oracle is the definition in the (blocknum, KV_N, blocksize, D) layout with
per-channel parameters: the layout only moves bytes, and per-tensor parameters are the
per-channel ones with every channel equal.  The variant runs must therefore also be bit
for bit those of the plain path on the same data.
"""
import zlib

import numpy as np
import pytest
import torch

import fia_workloads as W
import oracle as OR
from parity import (OUT_TOL, SUM_TOL, DeviceDecode, assert_close, assert_close_max, check_codes, compare_decode,
                    oracle_decode, run_decode)

pytestmark = pytest.mark.gpu

LAYOUT_CASES = {
    # name: make_decode_case kwargs; covers the bf16/fp16 tensor-core kernel (D 128, and D 64
    # stacked), the int8 tensor-core kernel (D 128) and the CUDA-core int8 kernel (D 64)
    "bf16_d128_g4": dict(B=3, Nq=8, Nkv=2, D=128, block_size=128, lengths=[300, 129, 1000]),
    "fp16_d64_g2_bs16": dict(B=2, Nq=4, Nkv=2, D=64, block_size=16, dtype=W.FP16, lengths=[77, 250]),
    "bf16_d64_g8_sink": dict(B=2, Nq=8, Nkv=1, D=64, block_size=64, lengths=[200, 31], sink=True),
    "int8_d128_g8": dict(B=2, Nq=16, Nkv=2, D=128, block_size=128, kv_dtype=W.INT8, lengths=[700, 130]),
    "int8_d64_g2": dict(B=2, Nq=4, Nkv=2, D=64, block_size=64, kv_dtype=W.INT8, lengths=[300, 65]),
}


def _case(name, **kw):
    return W.make_decode_case(seed=zlib.crc32(name.encode()) % (1 << 30), **kw)


def _bnbsh(cache: torch.Tensor) -> torch.Tensor:
    """(num_blocks, Nkv, block_size, D) -> (num_blocks, block_size, Nkv * D), same values."""
    nb, nkv, bs, d = cache.shape
    return cache.permute(0, 2, 1, 3).reshape(nb, bs, nkv * d).contiguous()


def _run(F, dd, ns=0, **kw):
    c = dd.case
    rows = (c.B, c.Nq) if kw.get("q_len", 1) <= 1 else (c.B, kw["q_len"], c.Nq)
    mx = torch.full(rows, float("nan"), dtype=torch.float32, device=dd.q.device)
    sm = torch.full(rows, float("nan"), dtype=torch.float32, device=dd.q.device)
    k, v = kw.pop("k", dd.k), kw.pop("v", dd.v)
    out, mx, sm = F.fia_decode_ex(dd.q, k, v, dd.bt, dd.lens, max_kv_len=c.max_len, num_heads=c.Nq,
                                  num_kv_heads=c.Nkv, scale=c.scale, antiquant_scale=kw.pop("aq_scale", dd.aq_scale),
                                  antiquant_offset=kw.pop("aq_offset", dd.aq_offset), sink=dd.sink,
                                  softmax_max=mx, softmax_sum=sm, num_splits=ns, **kw)
    return out, mx, sm


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("name", sorted(LAYOUT_CASES))
def test_bnbsh_layout(F, cuda, name, num_splits):
    case = _case(name, **LAYOUT_CASES[name])
    dd = DeviceDecode(case)
    out, mx, sm = _run(F, dd, num_splits, k=_bnbsh(dd.k), v=_bnbsh(dd.v), kv_layout=F.KV_BNBSH)
    compare_decode(case, out, mx, sm, ref=oracle_decode(case))
    base = run_decode(F, dd, num_splits=num_splits)
    assert torch.equal(out.view(torch.int16), base[0].view(torch.int16))
    assert torch.equal(mx, base[1]) and torch.equal(sm, base[2])
    assert F.fia_device_status() == 0


@pytest.mark.parametrize("D", [64, 128])
def test_int8_per_tensor_antiquant(F, cuda, D):
    name = f"per_tensor_d{D}"
    case = _case(name, B=3, Nq=8, Nkv=2, D=D, block_size=64, kv_dtype=W.INT8, lengths=[300, 77, 640])
    s2 = np.array([0.013, 0.007], np.float32)   # keys, values
    o2 = np.array([0.5, -1.25], np.float32)
    case.aq_scale = np.ascontiguousarray(np.broadcast_to(s2[:, None, None], (2, case.Nkv, D)), dtype=np.float32)
    case.aq_offset = np.ascontiguousarray(np.broadcast_to(o2[:, None, None], (2, case.Nkv, D)), dtype=np.float32)
    dd = DeviceDecode(case)
    for ns in (0, 2):
        out, mx, sm = _run(F, dd, ns, aq_scale=torch.from_numpy(s2).cuda(), aq_offset=torch.from_numpy(o2).cuda(),
                           antiquant_mode=F.AQ_PER_TENSOR)
        compare_decode(case, out, mx, sm, ref=oracle_decode(case))
        base = run_decode(F, dd, num_splits=ns)
        assert torch.equal(out.view(torch.int16), base[0].view(torch.int16))
    # without an offset
    out, mx, sm = _run(F, dd, aq_scale=torch.from_numpy(s2).cuda(), aq_offset=None, antiquant_mode=F.AQ_PER_TENSOR)
    case.aq_offset = None
    compare_decode(case, out, mx, sm, ref=oracle_decode(case))
    assert F.fia_device_status() == 0


def test_per_tensor_antiquant_needs_int8(F, cuda):
    case = _case("per_tensor_bf16", B=1, Nq=2, Nkv=1, D=64, block_size=16, lengths=[20])
    dd = DeviceDecode(case)
    s2 = torch.ones(2, dtype=torch.float32, device="cuda")
    with pytest.raises(F.FiaError):
        _run(F, dd, aq_scale=s2, antiquant_mode=F.AQ_PER_TENSOR)


@pytest.mark.parametrize("sink", [False, True])
@pytest.mark.parametrize("with_max_sum", [False, True])
def test_softmax_lse(F, cuda, sink, with_max_sum):
    """lse = ln(sum_t e^{z_t} (+ e^{s_h})) = M + ln(W) from the oracle's M and W; a row with
    neither a visible key nor a sink gives -inf (batch 1 is empty)."""
    case = _case(f"lse_{sink}", B=3, Nq=4, Nkv=2, D=128, block_size=128, lengths=[200, 0, 1500], sink=sink)
    dd = DeviceDecode(case)
    lse = torch.full((case.B, case.Nq), float("nan"), dtype=torch.float32, device="cuda")
    c = case
    kw = {}
    if with_max_sum:
        kw = dict(softmax_max=torch.empty((c.B, c.Nq), dtype=torch.float32, device="cuda"),
                  softmax_sum=torch.empty((c.B, c.Nq), dtype=torch.float32, device="cuda"))
    F.fia_decode_ex(dd.q, dd.k, dd.v, dd.bt, dd.lens, max_kv_len=c.max_len, num_heads=c.Nq, num_kv_heads=c.Nkv,
                    scale=c.scale, sink=dd.sink, softmax_lse=lse, **kw)
    _, m_ref, s_ref = oracle_decode(case)
    with np.errstate(divide="ignore"):
        lse_ref = np.where(s_ref > 0, m_ref + np.log(s_ref), -np.inf)
    got = lse.double().cpu().numpy().reshape(-1)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.all(got[~fin] == -np.inf)
    assert_close_max("softmax_lse", got[fin], lse_ref[fin])
    assert F.fia_device_status() == 0


# ------------------------------------------------------------------ attenMask (B, 1, 1, S)
MASK_CASES = {
    # bf16/fp16 tensor-core kernel (D 128 and stacked D 64 with a sink), the int8 tensor-core
    # kernel (D 128) and the CUDA-core int8 kernel (D 64)
    "bf16_d128_g4": dict(B=4, Nq=8, Nkv=2, D=128, block_size=128, lengths=[700, 129, 1000, 300]),
    "fp16_d64_g8_sink": dict(B=3, Nq=8, Nkv=1, D=64, block_size=64, dtype=W.FP16, lengths=[450, 31, 260],
                             sink=True),
    "int8_d128_g8": dict(B=4, Nq=16, Nkv=2, D=128, block_size=128, kv_dtype=W.INT8, lengths=[900, 130, 600, 257]),
    "int8_d64_g2": dict(B=3, Nq=4, Nkv=2, D=64, block_size=64, kv_dtype=W.INT8, lengths=[300, 65, 190]),
}


def _mask_for(case, seed, S):
    """Random keys masked (about 30%), batch 1 fully masked, the first 256 keys of batch 0
    masked (whole leading tiles: no reference maximum yet) and batch 2's last tile masked."""
    rng = np.random.default_rng(seed)
    m = rng.random((case.B, S)) < 0.3
    m[1, :] = True
    m[0, :256] = True
    L2 = int(case.lengths[2])
    m[2, max(0, L2 - 100):] = True
    return m


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("name", sorted(MASK_CASES))
def test_atten_mask(F, cuda, name, num_splits):
    case = _case("mask_" + name, **MASK_CASES[name])
    dd = DeviceDecode(case)
    S = case.max_len + 40  # mask rows longer than max_kv_len
    m = _mask_for(case, zlib.crc32(name.encode()) & 0xffff, S)
    ref = oracle_decode(case, mask=m.astype(np.uint8))
    for dtype in (torch.bool, torch.uint8):
        mask = torch.from_numpy(m).to(dtype).reshape(case.B, 1, 1, S).cuda()
        out, mx, sm = _run(F, dd, num_splits, atten_mask=mask)
        compare_decode(case, out, mx, sm, ref=ref)
    # an all-zero mask is no mask, bit for bit
    zero = torch.zeros((case.B, S), dtype=torch.int8, device="cuda")
    out, mx, sm = _run(F, dd, num_splits, atten_mask=zero)
    base = run_decode(F, dd, num_splits=num_splits)
    assert torch.equal(out.view(torch.int16), base[0].view(torch.int16))
    assert torch.equal(mx, base[1]) and torch.equal(sm, base[2])
    assert F.fia_device_status() == 0


def _poison_keys(case, drop):
    """NaN into the K and V rows of every key t of batch b with drop(b, t) true."""
    k, v = case.k_cache.copy(), case.v_cache.copy()
    nan = W.NAN_BITS[case.kv_dtype]
    for b in range(case.B):
        for t in range(int(case.lengths[b])):
            if drop(b, t):
                blk, row = case.block_table[b, t // case.block_size], t % case.block_size
                k[blk, :, row] = nan
                v[blk, :, row] = nan
    case.k_cache, case.v_cache = k, v


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("name", ["bf16_d128_g4", "fp16_d64_g8_sink"])
def test_atten_mask_nan_in_masked_keys(F, cuda, name, num_splits):
    """A masked key contributes nothing even when its cache rows hold NaN (16-bit KV; int8
    codes cannot be NaN)."""
    case = _case("mask_" + name, **MASK_CASES[name])
    S = case.max_len + 40
    m = _mask_for(case, zlib.crc32(name.encode()) & 0xffff, S)
    ref = oracle_decode(case, mask=m.astype(np.uint8))
    _poison_keys(case, lambda b, t: m[b, t])
    dd = DeviceDecode(case)
    mask = torch.from_numpy(m).reshape(case.B, 1, 1, S).cuda()
    out, mx, sm = _run(F, dd, num_splits, atten_mask=mask)
    compare_decode(case, out, mx, sm, ref=ref)
    assert F.fia_device_status() == 0


@pytest.mark.parametrize("name", ["bf16_d128_g4", "fp16_d64_g8_sink"])
def test_decode_band_window_nan_outside(F, cuda, name):
    """Keys before the window (in the window's first tile and before it) hold NaN."""
    case = _case("window_" + name, **WINDOW_CASES[name])
    pre, nxt = 100, 0
    ref = oracle_decode(case, band=(pre, nxt))
    _poison_keys(case, lambda b, t: t < int(case.lengths[b]) - 1 - pre)
    dd = DeviceDecode(case)
    for ns in (0, 3):
        out, mx, sm = _run(F, dd, ns, pre_tokens=pre, next_tokens=nxt)
        compare_decode(case, out, mx, sm, ref=ref)
    assert F.fia_device_status() == 0


def test_atten_mask_rows_too_short(F, cuda):
    case = _case("mask_short", B=2, Nq=4, Nkv=2, D=128, block_size=128, lengths=[300, 20])
    dd = DeviceDecode(case)
    mask = torch.zeros((case.B, case.max_len - 1), dtype=torch.bool, device="cuda")
    with pytest.raises(F.FiaError):
        _run(F, dd, atten_mask=mask)


# ------------------------------------------------------------------ int8 post-quant output
PQ_CASES = {
    "bf16_d128_g4_empty": dict(B=4, Nq=8, Nkv=2, D=128, block_size=128, lengths=[700, 0, 1000, 129]),
    "fp16_d64_g8_sink": dict(B=3, Nq=8, Nkv=1, D=64, block_size=64, dtype=W.FP16, lengths=[450, 0, 260],
                             sink=True),
    "int8_d128_g8": dict(B=3, Nq=16, Nkv=2, D=128, block_size=128, kv_dtype=W.INT8, lengths=[900, 130, 0]),
    "int8_d64_g2": dict(B=2, Nq=4, Nkv=2, D=64, block_size=64, kv_dtype=W.INT8, lengths=[300, 65]),
}


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("name", sorted(PQ_CASES))
def test_post_quant_int8_output(F, cuda, name, num_splits):
    case = _case("pq_" + name, **PQ_CASES[name])
    dd = DeviceDecode(case)
    o_ref, m_ref, s_ref = oracle_decode(case)
    C = case.Nq * case.D
    rng = np.random.default_rng(zlib.crc32(name.encode()) & 0xffff)
    amax = max(float(np.abs(o_ref).max()), 1e-3)
    atol, rtol = OUT_TOL[case.dtype]
    per_channel = (rng.uniform(0.5, 1.5, C) * 60.0 / amax).astype(np.float32)
    offsets = rng.uniform(-20, 20, C).astype(np.float32)
    variants = [  # (scale2, offset2): per tensor / per channel, symmetric / asymmetric, saturating
        (np.array([60.0 / amax], np.float32), None),
        (np.array([60.0 / amax], np.float32), np.array([-7.5], np.float32)),
        (per_channel, None),
        (per_channel, offsets),
        (np.array([1000.0 / amax], np.float32), np.array([3.0], np.float32)),
    ]
    for s2, o2 in variants:
        y, _ = OR.post_quant(o_ref.reshape(case.B, C), s2, o2)   # channels h * D + d of a batch row
        out, mx, sm = _run(F, dd, num_splits, quant_scale2=torch.from_numpy(s2).cuda(),
                           quant_offset2=None if o2 is None else torch.from_numpy(o2).cuda())
        assert out.dtype == torch.int8 and tuple(out.shape) == (case.B, case.Nq, case.D)
        s_c = np.broadcast_to(s2.astype(np.float64), (C,))
        check_codes(out.cpu().numpy().reshape(-1, C), y.reshape(-1, C), o_ref.reshape(-1, C), s_c, atol, rtol)
        assert_close_max("softmax_max", mx.double().cpu().numpy().reshape(-1), m_ref)
        assert_close("softmax_sum", sm.double().cpu().numpy().reshape(-1), s_ref, *SUM_TOL)
    assert F.fia_device_status() == 0


def test_post_quant_offset_without_scale(F, cuda):
    case = _case("pq_bad", B=1, Nq=2, Nkv=1, D=64, block_size=16, lengths=[20])
    dd = DeviceDecode(case)
    with pytest.raises(F.FiaError):
        F.fia_decode_ex(dd.q, dd.k, dd.v, dd.bt, dd.lens, max_kv_len=case.max_len, num_heads=case.Nq,
                        num_kv_heads=case.Nkv, scale=case.scale, quant_offset2=torch.zeros(1, device="cuda"),
                        out=torch.empty((1, 2, 64), dtype=torch.int8, device="cuda"))


@pytest.mark.parametrize("D,num_splits", [(128, 0), (64, 0), (128, 2)])
def test_post_quant_ties_and_saturation_exact(F, cuda, D, num_splits):
    """Sequences of one key: the attention output is that key's value row, exactly in fp32.
    Values are multiples of 0.25 (exact in bf16), so with scale2 = 2 half of y = 2v + o
    fall on ties (rounded to even) and with scale2 = 4 the large ones saturate: the int8
    output must equal the oracle's codes bit for bit.  Batch 3 is empty: code = q(0)."""
    lengths = [1, 1, 1, 0, 1, 1]
    case = _case(f"pq_exact_{D}", B=6, Nq=8, Nkv=2, D=D, block_size=64, lengths=lengths)
    rng = np.random.default_rng(D)
    vals = rng.integers(-255, 256, case.v_cache.shape).astype(np.float32) * 0.25   # |v| <= 63.75
    case.v_cache = W.to_bits(vals, case.dtype)
    assert np.array_equal(W.bits_to_f32(case.v_cache, case.dtype), vals)
    dd = DeviceDecode(case)
    o_ref, _, _ = oracle_decode(case)
    for s2, o2 in [(2.0, 0.0), (2.0, 0.5), (4.0, -1.0), (0.5, 0.25)]:
        y, code_ref = OR.post_quant(o_ref.reshape(case.B, -1), [s2], [o2])
        out, _, _ = _run(F, dd, num_splits, quant_scale2=torch.tensor([s2], device="cuda"),
                         quant_offset2=torch.tensor([o2], device="cuda"))
        got = out.cpu().numpy().reshape(code_ref.shape)
        assert np.array_equal(got, code_ref), np.argwhere(got != code_ref)[:4].tolist()
        if s2 == 4.0:
            assert not np.any(y == np.floor(y) + 0.5)
        else:
            assert np.any(y == np.floor(y) + 0.5)      # ties present
        if s2 == 4.0:
            assert np.any(code_ref == 127) and np.any(code_ref == -128)
    assert F.fia_device_status() == 0


# ------------------------------------------------------------------ band window (one query)
WINDOW_CASES = {
    "bf16_d128_g4": dict(B=4, Nq=8, Nkv=2, D=128, block_size=128, lengths=[700, 129, 1000, 3]),
    "fp16_d64_g8_sink": dict(B=3, Nq=8, Nkv=1, D=64, block_size=64, dtype=W.FP16, lengths=[450, 31, 260],
                             sink=True),
    "int8_d128_g8": dict(B=3, Nq=16, Nkv=2, D=128, block_size=128, kv_dtype=W.INT8, lengths=[900, 130, 600]),
    "int8_d64_g2": dict(B=3, Nq=4, Nkv=2, D=64, block_size=32, kv_dtype=W.INT8, lengths=[300, 65, 190]),
}
WINDOWS = [(255, 0), (100, 0), (0, 0), (1000, -5), (7, -3), (130, 3)]


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("name", sorted(WINDOW_CASES))
def test_decode_band_window(F, cuda, name, num_splits):
    """Keys L - 1 - pre .. L - 1 + next: windows that start inside a tile, end before the
    last key, hold one key, or cover a whole short batch; chunked windows (splits 3)."""
    case = _case("window_" + name, **WINDOW_CASES[name])
    dd = DeviceDecode(case)
    for pre, nxt in WINDOWS:
        out, mx, sm = _run(F, dd, num_splits, pre_tokens=pre, next_tokens=nxt)
        compare_decode(case, out, mx, sm, ref=oracle_decode(case, band=(pre, nxt)))
    # a band wider than every sequence is no band, bit for bit
    out, mx, sm = _run(F, dd, num_splits, pre_tokens=1 << 40, next_tokens=1 << 40)
    base = run_decode(F, dd, num_splits=num_splits)
    assert torch.equal(out.view(torch.int16), base[0].view(torch.int16))
    assert torch.equal(mx, base[1]) and torch.equal(sm, base[2])
    assert F.fia_device_status() == 0


def test_decode_band_window_with_mask_and_int8_out(F, cuda):
    """The window composes with the attenMask and with the int8 output."""
    case = _case("window_mix", B=3, Nq=8, Nkv=2, D=128, block_size=64, lengths=[600, 200, 90])
    dd = DeviceDecode(case)
    S = case.max_len
    m = np.random.default_rng(5).random((case.B, S)) < 0.25
    mask = torch.from_numpy(m).cuda()
    out, mx, sm = _run(F, dd, 2, pre_tokens=300, next_tokens=0, atten_mask=mask)
    ref = oracle_decode(case, band=(300, 0), mask=m.astype(np.uint8))
    compare_decode(case, out, mx, sm, ref=ref)
    s2 = np.array([40.0 / max(float(np.abs(ref[0]).max()), 1e-3)], np.float32)
    y, _ = OR.post_quant(ref[0].reshape(case.B, -1), s2, None)
    code, _, _ = _run(F, dd, 2, pre_tokens=300, next_tokens=0, atten_mask=mask, quant_scale2=torch.from_numpy(s2).cuda())
    C = case.Nq * case.D
    check_codes(code.cpu().numpy().reshape(-1, C), y.reshape(-1, C), ref[0].reshape(-1, C),
                 np.broadcast_to(s2.astype(np.float64), (C,)), *OUT_TOL[case.dtype])
    assert F.fia_device_status() == 0


def test_decode_band_window_full_size_sampled(F, cuda):
    """A window of 1024 keys on the full-size bf16 GQA decode workload, sampled rows."""
    case = W.bf16_gqa_decode()
    dd = DeviceDecode(case)
    out, mx, sm = _run(F, dd, 0, pre_tokens=1023, next_tokens=0)
    rows = np.random.default_rng(9).choice(case.B * case.Nq, 96, replace=False)
    compare_decode(case, out, mx, sm, rows=rows, ref=oracle_decode(case, rows=rows, band=(1023, 0)))
    assert F.fia_device_status() == 0


def test_decode_band_rejects_empty_band(F, cuda):
    case = _case("window_bad", B=1, Nq=2, Nkv=1, D=64, block_size=16, lengths=[20])
    dd = DeviceDecode(case)
    with pytest.raises(F.FiaError):
        _run(F, dd, pre_tokens=2, next_tokens=-3)


# ------------------------------------------------------------------ several query positions (Q_S > 1)
QLEN_CASES = {
    # name: (make_decode_case kwargs with Nq = query heads, q_len); the 16-bit tensor-core kernel
    # (D 128 and stacked D 64), the int8 tensor-core kernel (D 128) and the CUDA-core int8 kernel
    "bf16_d128_g4_s4": (dict(B=3, Nq=8, Nkv=2, D=128, block_size=128, lengths=[300, 3, 1000]), 4),
    "fp16_d64_g2_s8_sink_bs16": (dict(B=2, Nq=4, Nkv=2, D=64, block_size=16, dtype=W.FP16, lengths=[77, 250],
                                      sink=True), 8),
    "bf16_d128_mqa_s16": (dict(B=2, Nq=1, Nkv=1, D=128, block_size=64, lengths=[129, 15]), 16),
    "int8_d128_g2_s4": (dict(B=2, Nq=4, Nkv=2, D=128, block_size=128, kv_dtype=W.INT8, lengths=[700, 130]), 4),
    "int8_d64_g2_s3": (dict(B=2, Nq=4, Nkv=2, D=64, block_size=64, kv_dtype=W.INT8, lengths=[300, 2]), 3),
}


def _qlen_case(name, kw, s):
    """A decode case with s query positions: q drawn as (B, s * Nq, D) and viewed as (B, s, Nq, D)."""
    kw = dict(kw)
    nq = kw.pop("Nq")
    case = _case("qlen_" + name, Nq=nq * s, **kw)
    case.Nq = nq
    case.q = case.q.reshape(case.B, s, nq, case.D)
    if case.sink is not None:
        case.sink = np.ascontiguousarray(case.sink[:nq])
    return case


@pytest.mark.parametrize("num_splits", [0, 3])
@pytest.mark.parametrize("name", sorted(QLEN_CASES))
def test_decode_several_query_positions(F, cuda, name, num_splits):
    """Q_S > 1 over the paged cache (FusedInferAttentionScore): the s positions of a batch are
    its last s, each seeing the keys up to its own position (a position before the first key
    gets the empty-row outputs); the oracle's q_len reading, every row."""
    kw, s = QLEN_CASES[name]
    case = _qlen_case(name, kw, s)
    dd = DeviceDecode(case)
    out, mx, sm = _run(F, dd, num_splits, q_len=s)
    assert out.shape == (case.B, s, case.Nq, case.D) and mx.shape == (case.B, s, case.Nq)
    code = {W.BF16: OR.BF16, W.FP16: OR.F16}
    kvc = OR.I8 if case.kv_dtype == W.INT8 else code[case.kv_dtype]
    o_ref, m_ref, s_ref = OR.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=case.Nq, Nkv=case.Nkv,
                                    D=case.D, scale=case.scale, q_dtype=code[case.dtype], kv_dtype=kvc,
                                    block_table=case.block_table, block_size=case.block_size, aq_scale=case.aq_scale,
                                    aq_offset=case.aq_offset, sink=case.sink, q_len=s)
    assert_close("out", out.double().cpu().numpy().reshape(-1, case.D), o_ref, *OUT_TOL[case.dtype])
    assert_close_max("softmax_max", mx.double().cpu().numpy().reshape(-1), m_ref)
    assert_close("softmax_sum", sm.double().cpu().numpy().reshape(-1), s_ref, *SUM_TOL)
    assert F.fia_device_status() == 0


def test_decode_several_query_positions_lse_and_int8_out(F, cuda):
    """Q_S > 1 composed with the log-sum-exp and int8 outputs (every segment through the merge)."""
    case = _qlen_case("lse_q8", dict(B=2, Nq=8, Nkv=2, D=128, block_size=128, lengths=[500, 60]), 4)
    dd = DeviceDecode(case)
    lse = torch.empty((case.B, 4, case.Nq), dtype=torch.float32, device="cuda")
    out, mx, sm = _run(F, dd, 0, q_len=4, softmax_lse=lse)
    o_ref, m_ref, s_ref = OR.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=case.Nq, Nkv=case.Nkv,
                                    D=case.D, scale=case.scale, q_dtype=OR.BF16, kv_dtype=OR.BF16,
                                    block_table=case.block_table, block_size=case.block_size, q_len=4)
    fin = s_ref > 0
    assert_close_max("softmax_lse", lse.double().cpu().numpy().reshape(-1)[fin], (m_ref + np.log(s_ref))[fin])
    C = case.Nq * case.D
    s2 = np.array([50.0], np.float32)
    code, _, _ = _run(F, dd, 3, q_len=4, quant_scale2=torch.from_numpy(s2).cuda())
    assert code.dtype == torch.int8 and tuple(code.shape) == (case.B, 4, case.Nq, case.D)
    y, _ = OR.post_quant(o_ref.reshape(-1, C), s2)
    check_codes(code.cpu().numpy().reshape(-1, C), y.reshape(-1, C), o_ref.reshape(-1, C),
                 np.broadcast_to(s2.astype(np.float64), (C,)), *OUT_TOL[case.dtype])
    assert F.fia_device_status() == 0


def test_decode_several_query_positions_full_size(F, cuda):
    """The bf16 GQA decode workload with 4 query positions per batch (16 virtual heads per kv
    head), sampled rows: the cache is read once for the 4 positions."""
    base = W.bf16_gqa_decode()
    case = _qlen_case("full", dict(B=base.B, Nq=base.Nq, Nkv=base.Nkv, D=base.D, block_size=base.block_size,
                                   lengths=base.lengths), 4)
    dd = DeviceDecode(case)
    out, mx, sm = _run(F, dd, 0, q_len=4)
    rng = np.random.default_rng(12)
    rows = np.sort(rng.choice(case.B * 4 * case.Nq, size=512, replace=False)).astype(np.int64)
    o_ref, m_ref, s_ref = OR.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=case.Nq, Nkv=case.Nkv,
                                    D=case.D, scale=case.scale, q_dtype=OR.BF16, kv_dtype=OR.BF16,
                                    block_table=case.block_table, block_size=case.block_size, q_len=4, rows=rows)
    assert_close("out", out.double().cpu().numpy().reshape(-1, case.D)[rows], o_ref, *OUT_TOL[case.dtype])
    assert_close_max("softmax_max", mx.double().cpu().numpy().reshape(-1)[rows], m_ref)
    assert_close("softmax_sum", sm.double().cpu().numpy().reshape(-1)[rows], s_ref, *SUM_TOL)
    assert F.fia_device_status() == 0
