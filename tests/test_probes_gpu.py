"""Bit-exact and bounded parts of the decode path, through probes that run the
attention kernels' own device code: the element-wise int8 antiquant step and the
block-table gather; and for the int8 tensor-core kernel (int8 KV, D = 128), which
moves the antiquant off the element, its code -> fp16 conversion (exact) and its
query operand q' = q * s_K split into two fp16 parts (bounded)."""
import numpy as np
import pytest
import torch

import fia_workloads as W
import oracle
from parity import DeviceDecode, dev_bits

pytestmark = pytest.mark.gpu


def test_dequant_bit_exact_all_codes_all_channels(F, cuda):
    case = W.int8_antiquant_decode()
    sc, off = case.aq_scale.reshape(-1), case.aq_offset.reshape(-1)          # 2 * Nkv * D channels
    codes = np.repeat(np.arange(-128, 128, dtype=np.int8)[:, None], sc.size, axis=1).reshape(-1)
    scales = np.tile(sc, 256)
    offsets = np.tile(off, 256)
    got = F.fia_debug_dequant(torch.from_numpy(codes).to(cuda), torch.from_numpy(scales).to(cuda),
                              torch.from_numpy(offsets).to(cuda)).cpu().numpy()
    ref = oracle.default().dequant_i8_array(codes, offsets, scales)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("make", [
    lambda: W.bf16_gqa_decode(),
    lambda: W.make_decode_case(B=3, Nq=4, Nkv=2, D=64, block_size=16, dtype=W.FP16, lengths=[1, 47, 130],
                               seed=31, spare_blocks=3),
    lambda: W.make_decode_case(B=2, Nq=8, Nkv=2, D=64, block_size=32, kv_dtype=W.INT8, lengths=[33, 300], seed=37),
    lambda: W.make_decode_case(B=2, Nq=4, Nkv=2, D=128, block_size=48, lengths=[100, 47], seed=41),
], ids=["bf16_gqa_decode", "fp16_bs16", "int8_d64", "bs48"])
def test_gather_bit_exact(F, cuda, make):
    case = make()
    dd = DeviceDecode(case)
    rng = np.random.default_rng(7)
    pairs = {(int(np.argmax(case.lengths)), case.Nkv - 1), (int(np.argmin(case.lengths)), 0)}
    pairs |= {(int(rng.integers(case.B)), int(rng.integers(case.Nkv))) for _ in range(4)}
    for b, hk in sorted(pairs):
        L = int(case.lengths[b])
        got = F.fia_debug_gather(dd.k, dd.bt, dd.lens, max_kv_len=case.max_len, b=b, hkv=hk, length=L)
        ref = oracle.default().gather_rows(case.k_cache, case.block_table, b, hk, L, case.block_size)
        g = got.cpu().view(torch.int8 if case.kv_dtype == W.INT8 else torch.int16).numpy()
        assert np.array_equal(g.view(ref.dtype), ref), (b, hk)


def test_i8tc_code_conversion_bit_exact_all_codes(F, cuda):
    """Every code at every byte position of a 32-bit word becomes the fp16 of its value."""
    base = np.arange(-128, 128, dtype=np.int8)
    codes = np.stack([np.roll(base, k) for k in range(4)], axis=1).reshape(-1)
    got = F.fia_debug_i8_codes(torch.from_numpy(codes).to(cuda)).cpu().numpy().view(np.uint16)
    ref = codes.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("k_scale", [1.0, 1e4, 1e-6])
def test_i8tc_query_operand_split(F, cuda, k_scale):
    """hi + lo reproduces q * s_K (times a power of two) to 2^-21 of each head's largest
    entry (plus the fp32 product's own rounding, 2^-24), over the int8 workload's scales
    and scales 1e4 / 1e-6 times larger; the largest entry sits in [2^14, 2^15); the
    offset constant nq matches -scale log2(e) sum_d q_d s_d o_d; padded heads are zero."""
    case = W.int8_antiquant_decode()
    sc = case.aq_scale.copy()
    sc[0] *= np.float32(k_scale)
    scale = case.scale / k_scale
    B, Nq, Nkv, D = case.B, case.Nq, case.Nkv, case.D
    G = Nq // Nkv
    hi, lo, kn = F.fia_debug_i8_qprep(dev_bits(case.q, case.dtype, cuda), torch.from_numpy(sc).to(cuda),
                                      torch.from_numpy(case.aq_offset).to(cuda), num_heads=Nq, num_kv_heads=Nkv,
                                      scale=scale)
    hi = hi.cpu().numpy().view(np.float16).astype(np.float64)
    lo = lo.cpu().numpy().view(np.float16).astype(np.float64)
    kn = kn.cpu().numpy().astype(np.float64)
    assert not hi[:, :, G:].any() and not lo[:, :, G:].any() and not kn[:, :, G:].any()
    q = W.bits_to_f32(case.q, case.dtype).astype(np.float64).reshape(B, Nkv, G, D)
    qs = q * sc[0].astype(np.float64)[None, :, None, :]          # exact in fp64
    amax = np.abs(qs).max(axis=-1)                                # (B, Nkv, G)
    assert (amax > 0).all()
    v = hi[:, :, :G] + lo[:, :, :G]                               # exact in fp64
    vmax = np.abs(v).max(axis=-1)
    assert ((vmax >= 2.0 ** 14) & (vmax < 2.0 ** 15)).all()
    scale_log2 = float(np.float32(scale * 1.4426950408889634))
    p2 = kn[:, :, :G, 0] / scale_log2                             # 2^-e, exactly a power of two
    mant, _ = np.frexp(p2)
    assert (mant == 0.5).all()
    err = np.abs(v * p2[..., None] - qs).max(axis=-1)
    assert (err <= (2.0 ** -21 + 2.0 ** -24) * amax).all(), float((err / amax).max())
    o = case.aq_offset[0].astype(np.float64)[None, :, None, :]
    nq_ref = -scale_log2 * (qs * o).sum(axis=-1)
    nq_bound = 2.0 ** -19 * scale_log2 * np.abs(qs * o).sum(axis=-1)
    assert (np.abs(kn[:, :, :G, 1] - nq_ref) <= nq_bound).all()
