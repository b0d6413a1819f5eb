"""GPU parity of the context-parallel ring (attention_ifa_fia_gb300.ring.ring_decode_streams):
W ranks as CUDA streams of one GPU, each with one KV shard, partials passed around the ring
by device copies and merged by ring_attention_update; every rank's result is compared with
the oracle's attention over the unsplit cache (aclnnRingAttentionUpdate: merging the
partials of any split gives the unsplit result)."""
import zlib

import numpy as np
import pytest
import torch

import fia_workloads as W
from parity import DeviceDecode, compare_decode, oracle_decode, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def long_ctx(cuda):
    case = W.long_ctx_sink_decode()
    rows = sample_rows(case, 48, seed=8)
    return case, DeviceDecode(case), rows, oracle_decode(case, rows=rows)


@pytest.mark.parametrize("world", [2, 4, 8])
def test_ring_long_context_sink(F, long_ctx, world):
    """The long-context workload (B 4, 131072 keys, Nq 64, Nkv 8, D 64, sink) over 2, 4 and 8
    shards: every rank ends with the unsplit result, the sink counted once."""
    from attention_ifa_fia_gb300.ring import ring_decode_streams
    case, dd, rows, ref = long_ctx
    res = ring_decode_streams(dd.q, dd.k, dd.v, dd.bt, dd.lens, world=world, max_kv_len=case.max_len,
                              num_heads=case.Nq, num_kv_heads=case.Nkv, scale=case.scale, sink=dd.sink)
    torch.cuda.synchronize()
    for r in range(world):
        compare_decode(case, *res[r], rows=rows, ref=ref)
    assert F.fia_device_status() == 0


RING_CASES = {
    # name: (make_decode_case kwargs, worlds); shards past a short sequence's end give empty partials
    "ragged_bf16_g4": (dict(B=4, Nq=8, Nkv=2, D=128, block_size=64, lengths=[1000, 3, 257, 640], sink=True),
                       [1, 2, 3, 5]),
    "fp16_d64_bs16": (dict(B=3, Nq=4, Nkv=1, D=64, block_size=16, dtype=W.FP16, lengths=[300, 17, 0]), [2, 4]),
    "int8_d128_g8": (dict(B=2, Nq=16, Nkv=2, D=128, block_size=128, kv_dtype=W.INT8, lengths=[1500, 200]),
                     [2, 3]),
    "int8_d64": (dict(B=2, Nq=4, Nkv=2, D=64, block_size=32, kv_dtype=W.INT8, lengths=[333, 64]), [2]),
}


@pytest.mark.parametrize("name", sorted(RING_CASES))
def test_ring_cases(F, cuda, name):
    from attention_ifa_fia_gb300.ring import ring_decode_streams
    kw, worlds = RING_CASES[name]
    case = W.make_decode_case(seed=zlib.crc32(("ring_" + name).encode()) % (1 << 30), **kw)
    dd = DeviceDecode(case)
    ref = oracle_decode(case)
    for world in worlds:
        res = ring_decode_streams(dd.q, dd.k, dd.v, dd.bt, dd.lens, world=world, max_kv_len=case.max_len,
                                  num_heads=case.Nq, num_kv_heads=case.Nkv, scale=case.scale,
                                  antiquant_scale=dd.aq_scale, antiquant_offset=dd.aq_offset, sink=dd.sink)
        torch.cuda.synchronize()
        for r in range(world):
            compare_decode(case, *res[r], ref=ref)
    assert F.fia_device_status() == 0


def test_ring_repeated_calls_on_the_same_streams(F, cuda):
    """Back-to-back rings on the same streams (buffers of one call reused by the next): the
    results stay those of a single call, bit for bit."""
    from attention_ifa_fia_gb300.ring import ring_decode_streams
    case = W.make_decode_case(B=2, Nq=8, Nkv=2, D=128, block_size=128, lengths=[2000, 900], seed=91)
    dd = DeviceDecode(case)
    streams = [torch.cuda.Stream() for _ in range(4)]
    kw = dict(world=4, max_kv_len=case.max_len, num_heads=case.Nq, num_kv_heads=case.Nkv, scale=case.scale,
              streams=streams)
    first = ring_decode_streams(dd.q, dd.k, dd.v, dd.bt, dd.lens, **kw)
    torch.cuda.synchronize()
    first = [tuple(t.clone() for t in p) for p in first]
    for _ in range(5):
        again = ring_decode_streams(dd.q, dd.k, dd.v, dd.bt, dd.lens, **kw)
    torch.cuda.synchronize()
    for a, b in zip(first, again):
        assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
        assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


def test_ring_graph_replay(F, cuda):
    """The ring captured in a CUDA graph gives the eager ring's results bit for bit, and a
    replay after new input contents gives the oracle's result for them."""
    from attention_ifa_fia_gb300.ring import RingDecodeGraph, ring_decode_streams
    case = W.make_decode_case(B=3, Nq=8, Nkv=2, D=64, block_size=64, lengths=[3000, 1, 700], sink=True, seed=93)
    dd = DeviceDecode(case)
    kw = dict(world=4, max_kv_len=case.max_len, num_heads=case.Nq, num_kv_heads=case.Nkv, scale=case.scale,
              sink=dd.sink)
    eager = ring_decode_streams(dd.q, dd.k, dd.v, dd.bt, dd.lens, **kw)
    torch.cuda.synchronize()
    eager = [tuple(t.clone() for t in p) for p in eager]
    g = RingDecodeGraph(dd.q, dd.k, dd.v, dd.bt, dd.lens, **kw)
    got = g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, got):
        assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
        assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    other = W.make_decode_case(B=3, Nq=8, Nkv=2, D=64, block_size=64, lengths=[3000, 1, 700], sink=True, seed=94)
    od = DeviceDecode(other)
    dd.q.copy_(od.q)
    dd.k.copy_(od.k)
    dd.v.copy_(od.v)
    dd.bt.copy_(od.bt)
    dd.sink.copy_(od.sink)
    got = g.replay()
    torch.cuda.synchronize()
    ref = oracle_decode(other)
    for r in range(4):
        compare_decode(other, *got[r], ref=ref)
    assert F.fia_device_status() == 0
