"""GPU parity of fia_decode against the oracle (through the C interface).

The four decode workloads run at full size and are compared on sampled rows
(every head of the shortest and longest sequence plus random rows); small cases
that span several tiles, ragged tails and the degenerate cases are compared on
every row.  Tolerances are those stated in tests/parity.py.
"""
import zlib

import numpy as np
import pytest
import torch

import fia_workloads as W
from parity import DeviceDecode, assert_close, compare_decode, oracle_decode, run_decode, sample_rows, to_f64

pytestmark = pytest.mark.gpu


def _status(F):
    return F.fia_device_status()


# ----------------------------------------------------------------------------- the workloads
def test_tiny_decode_fp16(F, cuda):
    case = W.tiny_decode()
    dd = DeviceDecode(case)
    out, mx, sm = run_decode(F, dd)
    compare_decode(case, out, mx, sm)
    assert _status(F) == 0


def test_bf16_gqa_decode_full_size(F, cuda):
    case = W.bf16_gqa_decode()
    dd = DeviceDecode(case)
    out, mx, sm = run_decode(F, dd)
    rows = sample_rows(case, 256, seed=1)
    compare_decode(case, out, mx, sm, rows=rows)
    assert _status(F) == 0


def test_int8_antiquant_decode_full_size(F, cuda):
    """The int8 workload runs on the tensor-core kernel, which applies the antiquant to the
    query and the output instead of each element; besides the stated tolerances, its
    scores are checked through the softmax maximum at 1e-5 relative."""
    case = W.int8_antiquant_decode()
    dd = DeviceDecode(case)
    out, mx, sm = run_decode(F, dd)
    rows = sample_rows(case, 128, seed=2)
    ref = oracle_decode(case, rows=rows)
    compare_decode(case, out, mx, sm, rows=rows, ref=ref)
    assert_close("softmax_max at 1e-5", to_f64(mx).reshape(-1)[rows], ref[1], 0.0, 1e-5)
    assert _status(F) == 0


@pytest.fixture(scope="module")
def long_ctx(cuda):
    case = W.long_ctx_sink_decode()
    return case, DeviceDecode(case)


@pytest.mark.parametrize("num_splits", [W.LONG_CTX_CHUNKS, 0])
def test_long_ctx_sink_full_size(F, long_ctx, num_splits):
    case, dd = long_ctx
    out, mx, sm = run_decode(F, dd, num_splits=num_splits)
    rows = sample_rows(case, 48, seed=3)
    compare_decode(case, out, mx, sm, rows=rows)
    assert _status(F) == 0


def test_long_ctx_public_chunks_merged_by_rau(F, long_ctx):
    """The 32-chunk split done through the public API: one fia_decode per 4096-token chunk
    (the sink given to the first chunk only), folded in place by ring_attention_update."""
    case, dd = long_ctx
    n = W.LONG_CTX_CHUNKS
    chunk = case.max_len // n
    cols = chunk // case.block_size
    lens = torch.full((case.B,), chunk, dtype=torch.int64, device=dd.q.device)
    acc = None
    for j in range(n):
        bt = dd.bt[:, j * cols:(j + 1) * cols].contiguous()
        part = run_decode(F, dd, sink=dd.sink if j == 0 else None, max_kv_len=chunk, lens=lens, bt=bt)
        if acc is None:
            acc = part
        else:
            F.ring_attention_update(acc[0], acc[1], acc[2], part[0], part[1], part[2],
                                    out=acc[0], max_out=acc[1], sum_out=acc[2])
    rows = sample_rows(case, 48, seed=4)
    compare_decode(case, *acc, rows=rows)
    assert _status(F) == 0


# ----------------------------------------------------------------------------- small cases, every row
EDGE = {
    # name: (make_decode_case kwargs, num_splits list)
    "len1": (dict(B=3, Nq=4, Nkv=2, D=64, block_size=16, lengths=[1, 1, 1]), [0]),
    "blocks_exact": (dict(B=2, Nq=8, Nkv=2, D=128, block_size=128, lengths=[128, 256]), [0, 1, 3]),
    "blocks_pm1": (dict(B=3, Nq=8, Nkv=2, D=128, block_size=128, lengths=[127, 129, 255]), [0, 2]),
    "tiles_g1_fp16": (dict(B=4, Nq=4, Nkv=4, D=64, block_size=32, dtype=W.FP16, lengths=[63, 64, 65, 1000]),
                      [0, 1, 5]),
    "mqa_g8": (dict(B=2, Nq=8, Nkv=1, D=128, block_size=64, lengths=[300, 77]), [0, 4]),
    "g3_fp16": (dict(B=2, Nq=6, Nkv=2, D=64, block_size=16, dtype=W.FP16, lengths=[50, 33]), [0]),
    "g2_d128": (dict(B=2, Nq=4, Nkv=2, D=128, block_size=16, lengths=[200, 9]), [0, 7]),
    "empty_seqs": (dict(B=3, Nq=4, Nkv=2, D=64, block_size=16, lengths=[0, 17, 0]), [0]),
    "empty_seqs_sink": (dict(B=3, Nq=4, Nkv=2, D=64, block_size=16, lengths=[0, 17, 0], sink=True), [0]),
    "bs512": (dict(B=2, Nq=4, Nkv=2, D=128, block_size=512, lengths=[700, 1500]), [0, 3]),
    "bs48": (dict(B=2, Nq=4, Nkv=2, D=64, block_size=48, lengths=[100, 47]), [0]),
    "poisoned_pool": (dict(B=3, Nq=8, Nkv=2, D=128, block_size=128, lengths=[5, 130, 257], poison=True,
                           spare_blocks=3, table_pad=2), [0, 2]),
    "poisoned_bs16_fp16": (dict(B=2, Nq=4, Nkv=1, D=64, block_size=16, dtype=W.FP16, lengths=[31, 70],
                                poison=True, spare_blocks=2, table_pad=1), [0]),
    "int8_d64": (dict(B=2, Nq=8, Nkv=2, D=64, block_size=32, kv_dtype=W.INT8, lengths=[33, 200]), [0, 3]),
    "int8_fp16q_g4": (dict(B=2, Nq=4, Nkv=1, D=128, block_size=64, dtype=W.FP16, kv_dtype=W.INT8,
                           lengths=[100, 64], poison=True), [0]),
    "int8_nkv16": (dict(B=1, Nq=16, Nkv=16, D=64, block_size=32, kv_dtype=W.INT8, lengths=[70]), [0]),
    # int8 KV with D = 128 runs on the tensor-core kernel with the antiquant folded into q and out
    "int8_tc_ragged_g8": (dict(B=3, Nq=16, Nkv=2, D=128, block_size=128, kv_dtype=W.INT8, lengths=[1, 129, 700]),
                          [0, 1, 3]),
    "int8_tc_g1_bs32_fp16": (dict(B=2, Nq=4, Nkv=4, D=128, block_size=32, dtype=W.FP16, kv_dtype=W.INT8,
                                  lengths=[31, 300]), [0, 2]),
    "int8_tc_g2_bs256": (dict(B=2, Nq=4, Nkv=2, D=128, block_size=256, kv_dtype=W.INT8, lengths=[255, 1000]),
                         [0, 4]),
    "int8_tc_g3": (dict(B=2, Nq=6, Nkv=2, D=128, block_size=64, kv_dtype=W.INT8, lengths=[64, 191]), [0]),
    "int8_tc_poisoned_g8": (dict(B=3, Nq=8, Nkv=1, D=128, block_size=64, kv_dtype=W.INT8, lengths=[5, 130, 257],
                                 poison=True, spare_blocks=3, table_pad=2), [0, 2]),
    "int8_tc_empty_seqs": (dict(B=3, Nq=8, Nkv=2, D=128, block_size=32, kv_dtype=W.INT8, lengths=[0, 40, 0]), [0]),
    "int8_tc_one_tile_items": (dict(B=4, Nq=8, Nkv=2, D=128, block_size=64, kv_dtype=W.INT8, lengths=[1, 60, 128, 5]),
                               [0]),
    "one_tile_items_bf16": (dict(B=4, Nq=8, Nkv=2, D=128, block_size=64, lengths=[1, 60, 128, 5]), [0]),
    "int8_tc_many_batches": (dict(B=200, Nq=8, Nkv=2, D=128, block_size=128, kv_dtype=W.INT8, len_range=(0, 300)),
                             [0]),
    "sink_bf16": (dict(B=2, Nq=8, Nkv=2, D=64, block_size=16, lengths=[40, 90], sink=True), [0, 3]),
    "sink_fp16_d128": (dict(B=1, Nq=4, Nkv=4, D=128, block_size=128, dtype=W.FP16, lengths=[300], sink=True),
                       [0]),
    "many_batches": (dict(B=300, Nq=2, Nkv=1, D=64, block_size=16, len_range=(0, 40)), [0]),
    "batches_over_1024": (dict(B=1500, Nq=2, Nkv=2, D=64, block_size=16, dtype=W.FP16, len_range=(0, 20)), [0]),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_case(F, cuda, name):
    kw, splits = EDGE[name]
    case = W.make_decode_case(seed=zlib.crc32(name.encode()) % (1 << 30), **kw)
    dd = DeviceDecode(case)
    ref = oracle_decode(case)
    for ns in splits:
        out, mx, sm = run_decode(F, dd, num_splits=ns)
        compare_decode(case, out, mx, sm, ref=ref)
    assert _status(F) == 0


def test_int8_without_offset(F, cuda):
    """antiquant_offset may be omitted (treated as 0), on both int8 kernels."""
    for D in (64, 128):
        case = W.make_decode_case(B=2, Nq=8, Nkv=2, D=D, block_size=64, kv_dtype=W.INT8, lengths=[100, 333], seed=23)
        case.aq_offset = None
        dd = DeviceDecode(case)
        for ns in (0, 3):
            out, mx, sm = run_decode(F, dd, num_splits=ns)
            compare_decode(case, out, mx, sm)
    assert _status(F) == 0


@pytest.mark.parametrize("k_scale", [1e4, 1e-6])
def test_int8_key_scale_extremes(F, cuda, k_scale):
    """Key scales far from 1 (the softmax scale compensating) move q * scale_k far from
    the fp16 range; the power-of-two prescale keeps the scores exact."""
    case = W.make_decode_case(B=2, Nq=16, Nkv=2, D=128, block_size=128, kv_dtype=W.INT8, lengths=[500, 77],
                              seed=29)
    case.aq_scale = case.aq_scale.copy()
    case.aq_scale[0] *= np.float32(k_scale)
    case.scale = case.scale / k_scale
    dd = DeviceDecode(case)
    out, mx, sm = run_decode(F, dd, num_splits=2)
    compare_decode(case, out, mx, sm)
    assert _status(F) == 0


def test_max_kv_len_zero(F, cuda):
    case = W.make_decode_case(B=2, Nq=4, Nkv=2, D=64, block_size=16, lengths=[0, 0], seed=5, spare_blocks=1)
    dd = DeviceDecode(case)
    out, mx, sm = run_decode(F, dd, max_kv_len=0)
    assert torch.all(out == 0) and torch.all(mx == -float("inf")) and torch.all(sm == 0)


def test_deterministic(F, cuda):
    case = W.make_decode_case(B=8, Nq=16, Nkv=4, D=128, block_size=128, len_range=(1, 3000), seed=11)
    dd = DeviceDecode(case)
    a = run_decode(F, dd)
    b = run_decode(F, dd)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x,
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y)


def test_bad_block_index_is_flagged_not_read(F, cuda):
    """An out-of-range block-table entry in use is skipped and reported, with no fault."""
    case = W.make_decode_case(B=2, Nq=4, Nkv=2, D=64, block_size=16, lengths=[40, 20], seed=13)
    dd = DeviceDecode(case)
    F.fia_device_status()
    bt = dd.bt.clone()
    bt[0, 1] = case.num_blocks + 5
    run_decode(F, dd, bt=bt)
    assert F.fia_device_status() & 2
    out, mx, sm = run_decode(F, dd)  # the untouched table still gives correct results
    compare_decode(case, out, mx, sm)
    assert F.fia_device_status() == 0


def test_length_above_bound_is_clamped(F, cuda):
    case = W.make_decode_case(B=2, Nq=4, Nkv=2, D=64, block_size=16, lengths=[40, 20], seed=17, table_pad=2)
    dd = DeviceDecode(case)
    F.fia_device_status()
    lens = dd.lens.clone()
    lens[1] = 10_000
    out, mx, sm = run_decode(F, dd, lens=lens, max_kv_len=40)
    assert F.fia_device_status() & 4
    # row 1 was clamped to 40 tokens: its first 20 are the real ones, the next 20 come from
    # blocks past its table (entries -1 there are skipped and flagged); row 0 is unaffected
    ref = oracle_decode(case, rows=np.arange(0, case.Nq))
    from parity import assert_close, OUT_TOL
    assert_close("out row 0", to_f64(out)[0], ref[0], *OUT_TOL[case.dtype])
    F.fia_device_status()


def test_int8_scores_rising_along_the_sequence(F, cuda):
    """Key codes aligned with the query and growing tile after tile make each 128-token
    tile's scores exceed the previous maximum by about 2^9: the int8 kernel must raise
    its reference maximum and rescale in the middle of an item (random inputs almost
    never reach that path).  Values stay random."""
    case = W.make_decode_case(B=2, Nq=8, Nkv=2, D=128, block_size=128, kv_dtype=W.INT8, lengths=[700, 450],
                              seed=11)
    G = case.Nq // case.Nkv
    q = W.bits_to_f32(case.q, case.dtype)                       # (B, Nq, D)
    case.aq_scale[0] = 0.005                                     # key scale
    case.aq_offset[0] = 0.0
    for b in range(case.B):
        for h in range(case.Nkv):
            sign = np.where(q[b, h * G:(h + 1) * G].sum(axis=0) >= 0, 1, -1).astype(np.int32)
            for t in range(int(case.lengths[b])):
                c = min(127, 2 + 14 * (t // 128))              # about 9.5 log2 units more per tile
                blk, row = case.block_table[b, t // case.block_size], t % case.block_size
                case.k_cache[blk, h, row] = (sign * c).astype(np.int8)
    dd = DeviceDecode(case)
    ref = oracle_decode(case)
    for ns in (0, 3):
        out, mx, sm = run_decode(F, dd, num_splits=ns)
        compare_decode(case, out, mx, sm, ref=ref)
    assert _status(F) == 0
