"""The context-parallel ring (attention_ifa_fia_gb300.ring) on the CPU: its schedule, and
the whole exchange between gloo ranks in separate processes, each holding one KV shard's
partial and merging what arrives (here with the oracle's RingAttentionUpdate, in fp64),
against the oracle's attention over the unsplit cache."""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest

import fia_workloads as W


def test_ring_schedule_delivers_every_partial_once():
    from attention_ifa_fia_gb300.ring import ring_steps
    for world in range(1, 9):
        for r in range(world):
            steps = ring_steps(world, r)
            assert [s for s, *_ in steps] == list(range(1, world))
            assert sorted(o for *_, o in steps) == sorted(set(range(world)) - {r})
            for s, dst, src, origin in steps:
                assert dst == (r + 1) % world and src == (r - 1) % world
                # what arrives at step s is what the sender received at step s - 1 (its own at s = 1)
                sender = dict((t, o) for t, _, _, o in ring_steps(world, src))
                assert origin == (src if s == 1 else sender[s - 1])
    with pytest.raises(ValueError):
        ring_steps(2, 2)


def test_shard_tables_cover_every_key_once():
    import torch
    from attention_ifa_fia_gb300.ring import shard_tables
    case = W.make_decode_case(B=3, Nq=4, Nkv=2, D=64, block_size=16, lengths=[100, 37, 0], seed=3)
    bt = torch.from_numpy(case.block_table)
    lens = torch.from_numpy(case.lengths)
    for world in (1, 2, 3, 5, 8):
        S, tables, shard_lens = shard_tables(bt, lens, world=world, max_kv_len=case.max_len, block_size=16)
        assert S % 16 == 0 and S * world >= case.max_len
        for b in range(case.B):
            keys = []
            for r in range(world):
                n = int(shard_lens[r][b])
                for t in range(n):
                    keys.append((int(tables[r][b, t // 16]), t % 16))
            want = [(int(case.block_table[b, t // 16]), t % 16) for t in range(int(case.lengths[b]))]
            assert keys == want


def _partial(case, S, r, world):
    """Rank r's partial: the oracle's attention over keys [r S, (r + 1) S), the sink on rank 0 only."""
    import oracle
    bs = case.block_size
    cols = S // bs
    bt = np.full((case.B, cols), -1, np.int32)
    part = case.block_table[:, r * cols:(r + 1) * cols]
    bt[:, :part.shape[1]] = part
    lens = np.clip(case.lengths - r * S, 0, S)
    out, mx, sm = oracle.decode(case.q, case.k_cache, case.v_cache, lens, Nq=case.Nq, Nkv=case.Nkv, D=case.D,
                                scale=case.scale, q_dtype=oracle.BF16, kv_dtype=oracle.BF16, block_table=bt,
                                block_size=bs, sink=case.sink if r == 0 else None)
    return out.reshape(case.B, case.Nq, case.D), mx.reshape(case.B, case.Nq), sm.reshape(case.B, case.Nq)


def _ring_rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from attention_ifa_fia_gb300.ring import DistExchange, ring_merge
        case = W.make_decode_case(B=3, Nq=8, Nkv=2, D=64, block_size=16, lengths=[150, 37, 96], sink=True, seed=77)
        S = -(-(-(-case.max_len // world)) // 16) * 16
        mine = tuple(torch.from_numpy(np.ascontiguousarray(x)) for x in _partial(case, S, rank, world))

        def merge(a, b):
            return tuple(torch.from_numpy(x) for x in oracle.rau(*(t.numpy() for t in a), *(t.numpy() for t in b)))

        got = ring_merge(mine, world=world, rank=rank, exchange=DistExchange(), merge=merge)
        q.put((rank, tuple(t.numpy() for t in got)))
    except Exception as e:  # report, so the parent fails with the reason instead of a timeout
        q.put((rank, repr(e)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ring_on_gloo_ranks_equals_unsplit(world):
    """Each of `world` CPU ranks ends with attention over the whole cache: one rank's shard
    is past the shortest sequence's end (an empty partial), and the sink enters once."""
    import oracle
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ring_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    case = W.make_decode_case(B=3, Nq=8, Nkv=2, D=64, block_size=16, lengths=[150, 37, 96], sink=True, seed=77)
    ref = oracle.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=case.Nq, Nkv=case.Nkv, D=case.D,
                        scale=case.scale, q_dtype=oracle.BF16, kv_dtype=oracle.BF16, block_table=case.block_table,
                        block_size=case.block_size, sink=case.sink)
    for r in range(world):
        assert not isinstance(got[r], str), got[r]
        out, mx, sm = got[r]
        np.testing.assert_allclose(out.reshape(-1, case.D), ref[0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(mx.reshape(-1), ref[1], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(sm.reshape(-1), ref[2], rtol=1e-12)
