"""GPU parity of the decode variants of fia_decode_ex against the oracle.

aclnnIncreFlashAttentionV3, "Constraints / page attention": besides (blocknum, KV_N,
blocksize, D), the paged cache may be laid out (blocknum, blocksize, H), H = KV_N * D;
"antiquantScale / antiquantOffset": a per-tensor form of shape (2).
FusedInferAttentionScore: the softmaxLse output, ln of the softmax denominator.

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
from parity import MAX_TOL, DeviceDecode, assert_close, compare_decode, oracle_decode, run_decode

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
    mx = torch.full((c.B, c.Nq), float("nan"), dtype=torch.float32, device=dd.q.device)
    sm = torch.full((c.B, c.Nq), float("nan"), dtype=torch.float32, device=dd.q.device)
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
    assert_close("softmax_lse", got[fin], lse_ref[fin], *MAX_TOL)
    assert F.fia_device_status() == 0
