"""The seeded input recipes (fia_workloads.py) hold the properties the measurements and parity
tests rely on: shapes, length ranges, a pool of exactly sum ceil(L / blockSize) blocks (the
pages' BlockNum rule) used once each through the block table, -1 table padding, value
ranges of the int8 codes and antiquant parameters, exact storage rounding, determinism."""
import numpy as np
import pytest

import fia_workloads as W


def _check_pool(case):
    bs = case.block_size
    nblk = [(int(L) + bs - 1) // bs for L in case.lengths]
    assert case.num_blocks >= sum(nblk) == W.pool_blocks(case.lengths, bs)
    used = np.concatenate([case.block_table[b, :n] for b, n in enumerate(nblk)])
    assert len(np.unique(used)) == len(used) and used.min(initial=0) >= 0 and used.max(initial=0) < case.num_blocks
    for b, n in enumerate(nblk):
        assert np.all(case.block_table[b, n:] == -1)
    assert case.block_table.shape[1] >= max(max(nblk), 1)


@pytest.mark.parametrize("name,B,Nq,Nkv,D,lo,hi", [
    ("tiny_decode", 2, 4, 2, 64, 37, 100),
    ("bf16_gqa_decode", 32, 32, 8, 128, 1, 4096),
    ("int8_antiquant_decode", 64, 64, 8, 128, 512, 8192),
])
def test_decode_workload_recipe(name, B, Nq, Nkv, D, lo, hi):
    case = W.WORKLOADS[name]()
    assert (case.B, case.Nq, case.Nkv, case.D) == (B, Nq, Nkv, D)
    assert case.lengths.dtype == np.int64 and case.lengths.min() >= lo and case.lengths.max() <= hi
    assert case.q.shape == (B, Nq, D)
    assert case.k_cache.shape == case.v_cache.shape == (case.num_blocks, Nkv, case.block_size, D)
    _check_pool(case)
    if case.kv_dtype == W.INT8:
        assert case.k_cache.dtype == np.int8 and case.k_cache.min() >= -127 and case.k_cache.max() <= 127
        assert case.aq_scale.shape == case.aq_offset.shape == (2, Nkv, D)
        assert case.aq_scale.min() >= 0.005 and case.aq_scale.max() <= 0.02
        assert case.aq_offset.min() >= -2.0 and case.aq_offset.max() <= 2.0
    else:
        f = W.bits_to_f32(case.k_cache, case.kv_dtype)
        assert np.array_equal(W.to_bits(f, case.kv_dtype), case.k_cache)   # exact storage values
        tol = 5.0 / np.sqrt(f.size)                 # five standard errors of N(0, 1) statistics
        assert abs(float(f.mean())) < tol and abs(float(f.std()) - 1.0) < 4 * tol
    again = W.WORKLOADS[name]()
    assert np.array_equal(again.q, case.q) and np.array_equal(again.block_table, case.block_table)


def test_long_context_recipe_without_generating_it():
    """The long-context workload's shape is checked on its length rule alone (its cache is
    a gigabyte): 4 sequences of 131072 tokens split into 32 merged chunks."""
    assert W.LONG_CTX_CHUNKS == 32
    assert W.pool_blocks([131072] * 4, 128) == 4 * 1024


@pytest.mark.parametrize("name", ["causal_prefill_tnd", "causal_prefill_tnd_t8k"])
def test_prefill_workload_recipe(name):
    case = W.WORKLOADS[name]()
    assert (case.B, case.Nq, case.Nkv, case.D) == (8, 32, 8, 128)
    assert case.lengths_q.min() >= 1 and case.lengths_q.max() <= 2048
    assert np.array_equal(case.lengths_q, case.lengths_kv)
    assert case.cu_q[0] == 0 and np.array_equal(np.diff(case.cu_q), case.lengths_q)
    assert case.q.shape == (int(case.cu_q[-1]), 32, 128) and case.k.shape == (int(case.cu_kv[-1]), 8, 128)


def test_poisoned_slots_are_exactly_the_unused_ones():
    case = W.make_decode_case(B=3, Nq=4, Nkv=2, D=16, block_size=8, lengths=[9, 0, 16], spare_blocks=2,
                              table_pad=1, poison=True, seed=3)
    _check_pool(case)
    f = W.bits_to_f32(case.k_cache, case.kv_dtype)
    used = np.zeros((case.num_blocks, case.block_size), bool)
    for b in range(case.B):
        for t in range(int(case.lengths[b])):
            used[case.block_table[b, t // 8], t % 8] = True
    nan = np.isnan(f).all(axis=(1, 3))          # (blocks, rows): every head and channel NaN
    assert np.array_equal(nan, ~used)


def test_nominal_size_prefill_is_the_first_seed_near_8192():
    """The T = 8192 variant is the first seed from 1004 whose draw totals within 2% of 8192."""
    totals = {seed: int(W.causal_prefill_tnd(seed).cu_q[-1]) for seed in range(1004, 1011)}
    assert [s for s, t in totals.items() if abs(t - 8192) <= 0.02 * 8192] == [1010]
    assert int(W.causal_prefill_tnd_t8k().cu_q[-1]) == totals[1010] == 8267
