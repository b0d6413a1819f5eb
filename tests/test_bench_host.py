"""Host-side checks of bench.py: the roofline numerators (algorithmic decode bytes and
causal prefill FLOPs) against brute force, the traffic entry's source-hash gate, the clock
summary, and the multi-rank path (max over ranks, rank 0 alone reporting) on two gloo
ranks on the CPU."""
import importlib.util
import multiprocessing as mp
import os
import socket
import types

import numpy as np
import pytest

import fia_workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_prefill_flops_counts_visible_pairs():
    """4 D Nq per visible (query, key) pair: the causal count equals the ones of a
    lower-triangular matrix shifted to the bottom-right diagonal (np.tril, k = Lkv - Lq)."""
    B = _bench()
    case = W.make_prefill_case(Nq=3, Nkv=1, D=128, lengths=[5, 1, 9, 4], lengths_kv=[5, 7, 3, 0], seed=1)
    pairs_causal = sum(int(np.tril(np.ones((lq, lk), bool), k=lk - lq).sum())
                       for lq, lk in zip(case.lengths_q.tolist(), case.lengths_kv.tolist()))
    pairs_full = int((case.lengths_q * case.lengths_kv).sum())
    assert B.prefill_flops(case, causal=True) == 4 * 128 * 3 * pairs_causal
    assert B.prefill_flops(case, causal=False) == 4 * 128 * 3 * pairs_full


def test_decode_bytes_by_hand():
    B = _bench()
    case = W.make_decode_case(B=2, Nq=4, Nkv=2, D=64, block_size=16, lengths=[17, 3], seed=2)
    kv = (17 + 3) * 2 * 2 * 64 * 2                    # K and V, Nkv heads, D channels, 2 bytes
    qo = 2 * 2 * 4 * 64 * 2                           # q and out
    bt = (2 + 1) * 4                                  # blocks in use, int32
    aux = 2 * 8 + 2 * 2 * 4 * 4                       # lengths, max and sum
    got = B.decode_bytes(case)
    assert got["kv"] == kv and got["total"] == kv + qo + bt + aux


def test_traffic_entry_is_gated_by_the_source_hash(monkeypatch):
    """A recorded DRAM-traffic figure is reported only while the kernel sources hash to the
    value recorded with it; with any other hash it is null."""
    import json
    B = _bench()
    with open(os.path.join(ROOT, "profiles", "kernel_traffic.json")) as f:
        rec = json.load(f)
    for w in B.TRAFFIC_SOURCES:
        entry = rec.get(w)
        if entry and entry.get("sources_sha1") == B.traffic_sha(w):
            assert B.load_traffic(w) == entry["bytes_per_launch"]
        else:
            assert B.load_traffic(w) is None
        if entry:
            monkeypatch.setattr(B, "traffic_sha", lambda _w, sha=entry["sources_sha1"]: sha)
            assert B.load_traffic(w) == entry["bytes_per_launch"]
    monkeypatch.setattr(B, "traffic_sha", lambda w: "000000000000")
    assert all(B.load_traffic(w) is None for w in B.TRAFFIC_SOURCES)


def test_clock_summary():
    B = _bench()
    s = B.ClockSampler(0)
    s.samples = [(10.0, 2070.0, 2070.0, "900", []), (10.5, 2040.0, 2070.0, "950", ["sw_power_cap"]),
                 (11.0, 2070.0, 2070.0, "960", []), (11.5, 1000.0, 2070.0, "100", ["hw_slowdown"])]
    inside = s.summary(9.9, 11.1)
    assert inside["sm_mhz"] == 2070.0 and inside["reasons"] == ["sw_power_cap"] and inside["samples"] == 3
    assert inside["window"] == "timed region"
    short = s.summary(11.05, 11.1)                    # fewer than 3 samples: the last second of warm-up too
    assert short["window"].startswith("timed region and") and short["samples"] == 2


def test_reference_arm_runs_on_rank_0_only():
    B = _bench()
    args = types.SimpleNamespace(workload="tiny_decode", steps=1, warmup=0)
    assert B.run_reference(args, rank=1, world=2) is None


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B = _bench()
        got = B.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")   # per-rank durations 10 and 15
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_on_two_gloo_ranks():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 15.0, 1: 15.0}
    B = _bench()
    assert B.max_over_ranks(3.5, None, "cpu") == 3.5
