"""GPU parity of fia_prefill (TND, causal varlen, tcgen05) against the oracle, and of the
band mask of fia_prefill_ex (FusedInferAttentionScore sparseMode 4, preTokens/nextTokens)."""
import zlib

import numpy as np
import pytest
import torch

import fia_workloads as W
import oracle as OR
from parity import (OUT_TOL, SUM_TOL, DevicePrefill, assert_close, assert_close_max, check_codes, compare_prefill,
                    oracle_prefill, run_prefill, sample_prefill_rows)

pytestmark = pytest.mark.gpu


def test_causal_prefill_full_size(F, cuda):
    case = W.causal_prefill_tnd()
    dp = DevicePrefill(case)
    out, mx, sm = run_prefill(F, dp)
    rows = sample_prefill_rows(case, 1024, seed=5)
    compare_prefill(case, out, mx, sm, rows=rows)
    assert F.fia_device_status() == 0


CASES = {
    # name: make_prefill_case kwargs (+ "causal")
    "one_tile_each": dict(Nq=4, Nkv=2, D=128, lengths=[1, 127, 128, 129]),
    "ragged_multi_tile": dict(Nq=8, Nkv=2, D=128, lengths=[300, 513, 5]),
    "zero_length_seqs": dict(Nq=4, Nkv=4, D=128, lengths=[2, 2, 0, 2, 2]),
    "q_shorter_than_kv": dict(Nq=4, Nkv=1, D=128, lengths=[100, 200, 7], lengths_kv=[300, 200, 135]),
    "q_longer_than_kv": dict(Nq=2, Nkv=2, D=128, lengths=[200, 130], lengths_kv=[70, 0]),
    "gqa8_fp16": dict(Nq=16, Nkv=2, D=128, lengths=[260, 40], dtype=W.FP16),
    "sink": dict(Nq=4, Nkv=2, D=128, lengths=[150, 290], sink=True),
    "sink_q_longer": dict(Nq=2, Nkv=1, D=128, lengths=[140], lengths_kv=[20], sink=True),
    "no_mask": dict(Nq=4, Nkv=2, D=128, lengths=[77, 260], causal=False),
    "no_mask_lq_ne_lkv": dict(Nq=2, Nkv=1, D=128, lengths=[33, 140], lengths_kv=[500, 1], causal=False),
    # more sequences than the plan stages at a time (256), short ones and a long tail
    "many_seqs": dict(Nq=2, Nkv=1, D=128, lengths=[(i * 37) % 23 for i in range(600)] + [300]),
    "many_seqs_g1": dict(Nq=1, Nkv=1, D=128, lengths=[(i * 11) % 19 for i in range(300)] + [260, 0]),
    # head dim 64 (aclnnIncreFlashAttentionV3 "Constraints": D up to 512; 64 and 128 here) on
    # both kernels (even and odd GQA groups)
    "d64_pair": dict(Nq=8, Nkv=2, D=64, lengths=[300, 513, 5, 128]),
    "d64_odd_g": dict(Nq=3, Nkv=1, D=64, lengths=[129, 260, 1]),
    "d64_q_shorter_fp16_sink": dict(Nq=4, Nkv=2, D=64, lengths=[100, 7], lengths_kv=[300, 135], dtype=W.FP16,
                                    sink=True),
    "d64_no_mask_odd_g": dict(Nq=5, Nkv=5, D=64, lengths=[77, 200], causal=False),
    "d64_zero_length_seqs": dict(Nq=4, Nkv=4, D=64, lengths=[2, 0, 130, 0]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_case(F, cuda, name):
    kw = dict(CASES[name])
    causal = kw.pop("causal", True)
    case = W.make_prefill_case(seed=zlib.crc32(name.encode()) % (1 << 30), **kw)
    dp = DevicePrefill(case)
    out, mx, sm = run_prefill(F, dp, causal=causal)
    compare_prefill(case, out, mx, sm, causal=causal)
    assert F.fia_device_status() == 0


def test_prefill_deterministic(F, cuda):
    case = W.make_prefill_case(Nq=8, Nkv=2, D=128, lengths=[700, 333, 1024], seed=3)
    dp = DevicePrefill(case)
    a = run_prefill(F, dp)
    b = run_prefill(F, dp)
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_prefill_rejects_bad_arguments(F, cuda):
    case = W.make_prefill_case(Nq=4, Nkv=2, D=128, lengths=[5], seed=4)
    dp = DevicePrefill(case)
    with pytest.raises(F.FiaError) as ei:
        F.fia_prefill(dp.q, dp.k, dp.v, dp.cu_q, dp.cu_kv, max_seqlen_q=5, max_seqlen_kv=5, num_heads=4,
                      num_kv_heads=2, mask=2)
    assert ei.value.code == 161002


def test_prefill_scores_rising_along_the_keys(F, cuda):
    """Queries along one direction u and keys along u with a norm growing with the key
    index: every 128-key tile raises a row's maximum by far more than 2^8, so the
    kernel's lazy O rescale runs on every tile of every row (random inputs rarely)."""
    case = W.make_prefill_case(Nq=4, Nkv=2, D=128, lengths=[600, 300], seed=21)
    rng = np.random.default_rng(21)
    u = np.where(rng.random(case.D) < 0.5, -1.0, 1.0).astype(np.float32)
    q = np.broadcast_to(u, (case.T, case.Nq, case.D)) * 0.5
    case.q[...] = W.to_bits(np.ascontiguousarray(q, dtype=np.float32), case.dtype)
    k = np.empty((case.Tkv, case.Nkv, case.D), np.float32)
    for b in range(case.B):
        for j in range(int(case.lengths_kv[b])):
            k[case.cu_kv[b] + j] = u * (1.0 + j / 32.0)
    case.k[...] = W.to_bits(k, case.dtype)
    dp = DevicePrefill(case)
    out, mx, sm = run_prefill(F, dp)
    compare_prefill(case, out, mx, sm)
    assert F.fia_device_status() == 0


# ------------------------------------------------------------------ band (sparseMode 4)
BAND_CASES = {
    # name: (make_prefill_case kwargs, (pre_tokens, next_tokens)); even G runs the head-pair
    # kernel, odd G the single-head one
    "sliding_256_pair": (dict(Nq=8, Nkv=2, D=128, lengths=[700, 300, 129]), (255, 0)),
    "sliding_100_odd_g": (dict(Nq=3, Nkv=1, D=128, lengths=[500, 260]), (99, 0)),
    "both_sides": (dict(Nq=4, Nkv=2, D=128, lengths=[400, 3]), (50, 70)),
    "diagonal_only": (dict(Nq=4, Nkv=2, D=128, lengths=[130, 257]), (0, 0)),
    "lq_ne_lkv": (dict(Nq=4, Nkv=1, D=128, lengths=[100, 300], lengths_kv=[400, 200]), (150, 20)),
    "previous_5_only": (dict(Nq=2, Nkv=2, D=128, lengths=[260, 40]), (5, -1)),
    "future_only_odd_g": (dict(Nq=1, Nkv=1, D=128, lengths=[300]), (-3, 10)),
    "fp16_sink": (dict(Nq=4, Nkv=2, D=128, lengths=[333, 129], dtype=W.FP16, sink=True), (63, 0)),
    "sink_odd_g": (dict(Nq=3, Nkv=3, D=128, lengths=[200], sink=True), (17, 2)),
    "many_short_seqs": (dict(Nq=2, Nkv=1, D=128, lengths=[(i * 37) % 23 for i in range(300)] + [300]), (10, 0)),
    "wide_band_no_mask": (dict(Nq=4, Nkv=2, D=128, lengths=[77, 260], lengths_kv=[90, 260]), (1 << 40, 1 << 40)),
    "d64_sliding_pair": (dict(Nq=8, Nkv=2, D=64, lengths=[700, 129]), (200, 0)),
    "d64_both_sides_odd_g": (dict(Nq=3, Nkv=1, D=64, lengths=[400, 60], lengths_kv=[450, 60]), (50, 70)),
}


@pytest.mark.parametrize("name", sorted(BAND_CASES))
def test_prefill_band(F, cuda, name):
    kw, band = BAND_CASES[name]
    case = W.make_prefill_case(seed=zlib.crc32(("band_" + name).encode()) % (1 << 30), **kw)
    dp = DevicePrefill(case)
    out, mx, sm = run_prefill(F, dp, band=band)
    compare_prefill(case, out, mx, sm, band=band)
    assert F.fia_device_status() == 0


@pytest.mark.parametrize("Nq", [8, 6])  # head-pair and single-head kernels
def test_prefill_band_wide_pre_is_causal(F, cuda, Nq):
    """band(2^40, 0) is the rightDownCausal mask (the kernels without a lower edge), and so
    is band(max Lkv - 1, 0), which runs the kernels with a lower edge that excludes no key:
    both bit for bit the causal result."""
    case = W.make_prefill_case(Nq=Nq, Nkv=2, D=128, lengths=[700, 333, 50], lengths_kv=[800, 333, 20], seed=41)
    dp = DevicePrefill(case)
    a = run_prefill(F, dp)
    for band in [(1 << 40, 0), (int(case.lengths_kv.max()) - 1, 0)]:
        b = run_prefill(F, dp, band=band)
        assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
        assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_prefill_band_full_size_sampled(F, cuda):
    """A causal sliding window of 512 keys on the full-size prefill workload, sampled rows."""
    case = W.causal_prefill_tnd()
    dp = DevicePrefill(case)
    out, mx, sm = run_prefill(F, dp, band=(511, 0))
    rows = sample_prefill_rows(case, 1024, seed=6)
    compare_prefill(case, out, mx, sm, rows=rows, band=(511, 0))
    assert F.fia_device_status() == 0


def test_prefill_band_rejects(F, cuda):
    case = W.make_prefill_case(Nq=4, Nkv=2, D=128, lengths=[5], seed=4)
    dp = DevicePrefill(case)
    with pytest.raises(F.FiaError) as ei:   # a band holding no key
        run_prefill(F, dp, band=(3, -4))
    assert ei.value.code == 161002
    with pytest.raises(F.FiaError) as ei:   # mask 4 without the band's options
        F.fia_prefill(dp.q, dp.k, dp.v, dp.cu_q, dp.cu_kv, max_seqlen_q=5, max_seqlen_kv=5, num_heads=4,
                      num_kv_heads=2, mask=4)
    assert ei.value.code == 161001


# ------------------------------------------------------------------ paged keys (chunked prefill)
def _paged_pool(case, block_size, layout, seed, poison=False):
    """The case's TND keys and values scattered into a shuffled pool with a few unused blocks;
    rows past a sequence's length hold finite garbage, or NaN with poison=True (a cache taken
    from uninitialised memory).  Returns device (k_pool, v_pool, block_table, seq_lens_kv)."""
    rng = np.random.default_rng(seed)
    nblk = [-(-int(L) // block_size) for L in case.lengths_kv]
    total = sum(nblk) + 3
    perm = rng.permutation(total)
    width = max(max(nblk), 1)
    bt = np.full((case.B, width + 1), -1, np.int32)     # entries past the used ones are never read
    shape = (total, case.Nkv, block_size, case.D)
    pools = []
    for src in (case.k, case.v):
        if poison:
            pool = np.full(shape, W.NAN_BITS[case.dtype], np.uint16)
        else:
            pool = W.to_bits(rng.standard_normal(shape, dtype=np.float32) * 3, case.dtype)
        n = 0
        for b in range(case.B):
            for i in range(nblk[b]):
                blk = int(perm[n + i])
                bt[b, i] = blk
                t0, t1 = i * block_size, min(int(case.lengths_kv[b]), (i + 1) * block_size)
                pool[blk, :, :t1 - t0, :] = src[case.cu_kv[b] + t0:case.cu_kv[b] + t1].transpose(1, 0, 2)
            n += nblk[b]
        if layout == "bsh":
            pool = np.ascontiguousarray(pool.transpose(0, 2, 1, 3).reshape(total, block_size, case.Nkv * case.D))
        pools.append(torch.from_numpy(pool.view(np.int16)).cuda().view(torch.bfloat16 if case.dtype == W.BF16
                                                                           else torch.float16))
    return pools[0], pools[1], torch.from_numpy(bt).cuda(), torch.from_numpy(case.lengths_kv.astype(np.int64)).cuda()


PAGED_CASES = {
    # name: (make_prefill_case kwargs, block_size, layout, band); the query chunk of each
    # sequence is its last Lq positions
    "chunk_after_context_pair": (dict(Nq=8, Nkv=2, D=128, lengths=[128, 300, 1], lengths_kv=[1000, 300, 257]),
                                 128, "bnnbsd", None),
    "chunk_odd_g_bs256": (dict(Nq=3, Nkv=1, D=128, lengths=[200, 64], lengths_kv=[700, 64]), 256, "bnnbsd", None),
    "bsh_layout_bs512": (dict(Nq=4, Nkv=2, D=128, lengths=[333, 17], lengths_kv=[1300, 600]), 512, "bsh", None),
    "paged_band_fp16_sink": (dict(Nq=4, Nkv=2, D=128, lengths=[150, 290], lengths_kv=[900, 290], dtype=W.FP16,
                                  sink=True), 128, "bnnbsd", (255, 0)),
    "empty_kv_sequence": (dict(Nq=2, Nkv=1, D=128, lengths=[40, 70], lengths_kv=[0, 500]), 128, "bnnbsd", None),
    # blocks smaller than a key tile: several boxes per 128-key tile, one block each
    # (aclnnIncreFlashAttentionV3, "Constraints / page attention": blockSize a multiple of 16)
    "bs16_pair": (dict(Nq=8, Nkv=2, D=128, lengths=[100, 37], lengths_kv=[700, 300]), 16, "bnnbsd", None),
    "bs32_odd_g_bsh": (dict(Nq=3, Nkv=1, D=128, lengths=[64, 200], lengths_kv=[500, 200]), 32, "bsh", None),
    "bs48_band": (dict(Nq=4, Nkv=2, D=128, lengths=[130, 20], lengths_kv=[600, 333]), 48, "bnnbsd", (199, 0)),
    "bs64_fp16_sink": (dict(Nq=4, Nkv=4, D=128, lengths=[129, 1], lengths_kv=[257, 1], dtype=W.FP16, sink=True),
                       64, "bnnbsd", None),
    "d64_bs16_pair": (dict(Nq=8, Nkv=2, D=64, lengths=[100, 64], lengths_kv=[450, 64]), 16, "bnnbsd", None),
    "d64_bs256_odd_g_bsh": (dict(Nq=3, Nkv=3, D=64, lengths=[77, 130], lengths_kv=[600, 130]), 256, "bsh", None),
}


@pytest.mark.parametrize("poison", [False, True], ids=["finite_garbage", "nan_poisoned"])
@pytest.mark.parametrize("name", sorted(PAGED_CASES))
def test_prefill_paged_keys(F, cuda, name, poison):
    """Paged keys give the oracle's result and, tile for tile the same arithmetic, the TND
    run's result bit for bit -- also when every pool row that holds no key of a sequence
    (unused blocks, rows of a last block past the length) is NaN."""
    kw, bs, layout, band = PAGED_CASES[name]
    case = W.make_prefill_case(seed=zlib.crc32(("paged_" + name).encode()) % (1 << 30), **kw)
    dp = DevicePrefill(case)
    kp, vp, bt, lens = _paged_pool(case, bs, layout, seed=zlib.crc32(name.encode()) & 0xffff, poison=poison)
    c = case
    mx = torch.full((c.T, c.Nq), float("nan"), dtype=torch.float32, device="cuda")
    sm = torch.full((c.T, c.Nq), float("nan"), dtype=torch.float32, device="cuda")
    out, mx, sm = F.fia_prefill(dp.q, kp, vp, dp.cu_q, None, max_seqlen_q=int(c.lengths_q.max()),
                                max_seqlen_kv=int(c.lengths_kv.max()), num_heads=c.Nq, num_kv_heads=c.Nkv,
                                scale=c.scale, mask=4 if band else 3, sink=dp.sink, softmax_max=mx, softmax_sum=sm,
                                pre_tokens=band[0] if band else None, next_tokens=band[1] if band else None,
                                block_table=bt, seq_lens_kv=lens, kv_layout=F.KV_BNBSH if layout == "bsh" else 0)
    compare_prefill(case, out, mx, sm, band=band)
    ref = run_prefill(F, dp, band=band)
    assert torch.equal(out.view(torch.int16), ref[0].view(torch.int16))
    assert torch.equal(mx, ref[1]) and torch.equal(sm, ref[2])
    assert F.fia_device_status() == 0


@pytest.mark.parametrize("bs", [8, 24, 1024])
def test_prefill_paged_rejects_block_sizes(F, cuda, bs):
    """blockSize must be a multiple of 16 up to 512."""
    case = W.make_prefill_case(Nq=4, Nkv=2, D=128, lengths=[5], lengths_kv=[100], seed=4)
    dp = DevicePrefill(case)
    kp = torch.zeros((8, 2, bs, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((1, 100 // bs + 1), dtype=torch.int32, device="cuda")
    lens = torch.tensor([100], dtype=torch.int64, device="cuda")
    with pytest.raises(F.FiaError) as ei:
        F.fia_prefill(dp.q, kp, kp, dp.cu_q, None, max_seqlen_q=5, max_seqlen_kv=100, num_heads=4, num_kv_heads=2,
                      block_table=bt, seq_lens_kv=lens)
    assert ei.value.code == 161002


# ------------------------------------------------------------------ int8 post-quant output
# quantScale2 / quantOffset2 (aclnnIncreFlashAttentionV3 parameter table; FusedInferAttentionScore
# takes the pair in both modes) on the prefill output: both kernels, D 64 and 128, band, sink
PQ_CASES = {
    "pair_bf16_d128": (dict(Nq=8, Nkv=2, D=128, lengths=[300, 0, 129, 700]), None),
    "odd_g_fp16_d128_sink": (dict(Nq=3, Nkv=1, D=128, lengths=[260, 77], dtype=W.FP16, sink=True), None),
    "pair_bf16_d64_band": (dict(Nq=4, Nkv=2, D=64, lengths=[400, 130]), (100, 0)),
    "odd_g_bf16_d64": (dict(Nq=3, Nkv=3, D=64, lengths=[333, 1]), None),
}


def _run_pq(F, dp, band, s2, o2):
    c = dp.case
    mx = torch.full((c.T, c.Nq), float("nan"), dtype=torch.float32, device="cuda")
    sm = torch.full((c.T, c.Nq), float("nan"), dtype=torch.float32, device="cuda")
    return F.fia_prefill(dp.q, dp.k, dp.v, dp.cu_q, dp.cu_kv, max_seqlen_q=int(c.lengths_q.max(initial=0)),
                         max_seqlen_kv=int(c.lengths_kv.max(initial=0)), num_heads=c.Nq, num_kv_heads=c.Nkv,
                         scale=c.scale, mask=3 if band is None else 4, sink=dp.sink, softmax_max=mx,
                         softmax_sum=sm, pre_tokens=None if band is None else band[0],
                         next_tokens=None if band is None else band[1], quant_scale2=torch.from_numpy(s2).cuda(),
                         quant_offset2=None if o2 is None else torch.from_numpy(o2).cuda())


@pytest.mark.parametrize("name", sorted(PQ_CASES))
def test_prefill_post_quant_int8_output(F, cuda, name):
    kw, band = PQ_CASES[name]
    case = W.make_prefill_case(seed=zlib.crc32(("pq_" + name).encode()) % (1 << 30), **kw)
    dp = DevicePrefill(case)
    o_ref, m_ref, s_ref = oracle_prefill(case, band=band)
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
        y, _ = OR.post_quant(o_ref.reshape(case.T, C), s2, o2)   # channels h * D + d of a token row
        out, mx, sm = _run_pq(F, dp, band, s2, o2)
        assert out.dtype == torch.int8 and tuple(out.shape) == (case.T, case.Nq, case.D)
        s_c = np.broadcast_to(s2.astype(np.float64), (C,))
        check_codes(out.cpu().numpy().reshape(-1, C), y.reshape(-1, C), o_ref.reshape(-1, C), s_c, atol, rtol)
        assert_close_max("softmax_max", mx.double().cpu().numpy().reshape(-1), m_ref)
        assert_close("softmax_sum", sm.double().cpu().numpy().reshape(-1), s_ref, *SUM_TOL)
    assert F.fia_device_status() == 0


@pytest.mark.parametrize("Nq,D", [(4, 128), (3, 128), (4, 64), (1, 64)])
def test_prefill_post_quant_ties_and_saturation_exact(F, cuda, Nq, D):
    """Sequences of one query and one key: each output row is that key's value row, exactly
    in fp32.  Values are multiples of 0.25 (exact in bf16), so with scale2 = 2 half of
    y = 2v + o fall on ties (rounded to even) and with scale2 = 4 the large ones saturate:
    the int8 output equals the oracle's codes bit for bit, on the head-pair kernel (even G)
    and the single-head one (odd G)."""
    case = W.make_prefill_case(Nq=Nq, Nkv=1, D=D, lengths=[1] * 40 + [0, 1], seed=D + Nq)
    rng = np.random.default_rng(D * 7 + Nq)
    vals = rng.integers(-255, 256, case.v.shape).astype(np.float32) * 0.25   # |v| <= 63.75
    case.v = W.to_bits(vals, case.dtype)
    assert np.array_equal(W.bits_to_f32(case.v, case.dtype), vals)
    dp = DevicePrefill(case)
    o_ref, _, _ = oracle_prefill(case)
    C = Nq * D
    for s2, o2 in [(2.0, 0.0), (2.0, 0.5), (4.0, -1.0), (0.5, 0.25)]:
        y, code_ref = OR.post_quant(o_ref.reshape(case.T, C), [s2], [o2])
        out, _, _ = _run_pq(F, dp, None, np.array([s2], np.float32), np.array([o2], np.float32))
        got = out.cpu().numpy().reshape(code_ref.shape)
        assert np.array_equal(got, code_ref), np.argwhere(got != code_ref)[:4].tolist()
        if s2 == 4.0:
            assert not np.any(y == np.floor(y) + 0.5)
            assert np.any(code_ref == 127) and np.any(code_ref == -128)
        else:
            assert np.any(y == np.floor(y) + 0.5)      # ties present
    assert F.fia_device_status() == 0


def test_small_cases_after_full_size_launches(F, cuda):
    """Small launches after full-size ones whose buffers were freed, with host work in between
    (as a test sequence has it): the small case's inputs, outputs and workspace reuse the large
    one's memory, and every SM's tensor and shared memory still holds the large launch's data;
    the small case must read none of it (each one checked on every row against the oracle)."""
    small = [("no_mask", dict(Nq=4, Nkv=2, D=128, lengths=[77, 260]), False, None),
             ("sliding_256_pair", dict(Nq=8, Nkv=2, D=128, lengths=[700, 300, 129]), True, (255, 0)),
             ("one_tile_each", dict(Nq=4, Nkv=2, D=128, lengths=[1, 127, 128, 129]), True, None)]
    big = W.causal_prefill_tnd()
    rows = sample_prefill_rows(big, 256, seed=9)
    refs = {}
    for _round in range(2):
        for name, kw, causal, band in small:
            dpb = DevicePrefill(big)
            for _ in range(2):
                res = run_prefill(F, dpb)
            compare_prefill(big, *res, rows=rows)  # host work between the launches
            del dpb, res                            # the small case may reuse this memory
            if name not in refs:
                case = W.make_prefill_case(seed=zlib.crc32(("after_" + name).encode()) % (1 << 30), **kw)
                refs[name] = (case, oracle_prefill(case, causal=causal, band=band))
            case, ref = refs[name]
            dp = DevicePrefill(case)
            out, mx, sm = run_prefill(F, dp, causal=causal, band=band)
            compare_prefill(case, out, mx, sm, ref=ref, causal=causal, band=band)
            del dp, out, mx, sm
    assert F.fia_device_status() == 0


@pytest.mark.parametrize("name", ["chunk_after_context_pair", "chunk_odd_g_bs256", "bs16_pair", "bs48_band"])
def test_prefill_paged_keys_int8_output(F, cuda, name):
    """The int8 output over paged keys (NaN in every pool row that holds no key): codes within
    the tolerance band of the oracle's, and bit for bit those of the TND run on the same data."""
    kw, bs, layout, band = PAGED_CASES[name]
    case = W.make_prefill_case(seed=zlib.crc32(("paged_pq_" + name).encode()) % (1 << 30), **kw)
    dp = DevicePrefill(case)
    kp, vp, bt, lens = _paged_pool(case, bs, layout, seed=zlib.crc32(name.encode()) & 0xffff, poison=True)
    o_ref, m_ref, s_ref = oracle_prefill(case, band=band)
    C = case.Nq * case.D
    rng = np.random.default_rng(zlib.crc32(("pq" + name).encode()) & 0xffff)
    s2 = (rng.uniform(0.5, 1.5, C) * 60.0 / max(float(np.abs(o_ref).max()), 1e-3)).astype(np.float32)
    o2 = rng.uniform(-20, 20, C).astype(np.float32)
    c = case
    qs, qo = torch.from_numpy(s2).cuda(), torch.from_numpy(o2).cuda()
    out, mx, sm = F.fia_prefill(dp.q, kp, vp, dp.cu_q, None, max_seqlen_q=int(c.lengths_q.max()),
                                max_seqlen_kv=int(c.lengths_kv.max()), num_heads=c.Nq, num_kv_heads=c.Nkv,
                                scale=c.scale, mask=4 if band else 3, sink=dp.sink,
                                softmax_max=torch.empty((c.T, c.Nq), dtype=torch.float32, device="cuda"),
                                softmax_sum=torch.empty((c.T, c.Nq), dtype=torch.float32, device="cuda"),
                                pre_tokens=band[0] if band else None, next_tokens=band[1] if band else None,
                                block_table=bt, seq_lens_kv=lens, kv_layout=F.KV_BNBSH if layout == "bsh" else 0,
                                quant_scale2=qs, quant_offset2=qo)
    assert out.dtype == torch.int8
    y, _ = OR.post_quant(o_ref.reshape(c.T, C), s2, o2)
    check_codes(out.cpu().numpy().reshape(-1, C), y.reshape(-1, C), o_ref.reshape(-1, C), s2.astype(np.float64),
                *OUT_TOL[c.dtype])
    assert_close_max("softmax_max", mx.double().cpu().numpy().reshape(-1), m_ref)
    assert_close("softmax_sum", sm.double().cpu().numpy().reshape(-1), s_ref, *SUM_TOL)
    tnd = _run_pq(F, dp, band, s2, o2)
    assert torch.equal(out, tnd[0])
    assert F.fia_device_status() == 0
