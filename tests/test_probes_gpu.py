"""Bit-exact parts of the decode path: the int8 antiquant step and the block-table
gather, through probes that use the attention kernel's own device code."""
import numpy as np
import pytest
import torch

import fia_workloads as W
import oracle
from parity import DeviceDecode

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
