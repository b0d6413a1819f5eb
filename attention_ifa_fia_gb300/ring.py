"""Context parallelism for decode: KV shards, partials passed around a ring and merged by
RingAttentionUpdate.

aclnnRingAttentionUpdate ("功能说明 / 计算公式") merges two attention results over disjoint
key sets by their softmax max and sum; the FusedInferAttentionScore article gives the
operator a softmaxLse output for RingAttention.  With a long KV cache split into W shards
(shard r = keys [r * S, (r + 1) * S)), each of W ranks holds one shard and the same
queries, computes its partial (out, softmax max, softmax sum) with fia_decode, and the
partials travel around a ring:

    step s = 1 .. W - 1:  rank r sends to rank r + 1 the partial it received at step
                          s - 1 (its own at s = 1), receives from rank r - 1 the partial
                          of rank r - s, and merges it into its accumulator.

After W - 1 steps every rank holds the merge of all W partials, which equals attention
over the whole cache (the merge of the partials of any split is the unsplit result).  A
learnable sink belongs to the softmax once: only rank 0's fia_decode receives it.

Two drivers share the schedule (ring_steps):
  * ring_merge, for one process per rank: the exchange is a callable; DistExchange sends
    and receives through torch.distributed point-to-point operations (NCCL between GPUs,
    gloo between CPU processes), and the merge is ring_attention_update.
  * ring_decode_streams, one GPU: the W ranks are W CUDA streams, each rank's buffers its
    own device tensors, each send a device copy into the receiver's buffer, ordered by
    events (no kernel waits on another).  Every step's arithmetic runs in the library's
    kernels (fia_decode, ring_attention_update).
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import torch

from ._binding import fia_decode, fia_decode_workspace_size, ring_attention_update

Partial = Tuple[torch.Tensor, torch.Tensor, torch.Tensor]  # (out (rows, N, D), max (rows, N), sum (rows, N))


def ring_steps(world: int, rank: int) -> List[Tuple[int, int, int, int]]:
    """The ring schedule of one rank: (step, send_to, recv_from, origin) for steps 1 .. world - 1,
    origin being the rank whose partial arrives at that step."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a ring of {world}")
    return [(s, (rank + 1) % world, (rank - 1) % world, (rank - s) % world) for s in range(1, world)]


def rau_merge(acc: Partial, part: Partial) -> Partial:
    """acc merged with part by ring_attention_update (new tensors)."""
    return ring_attention_update(*acc, *part)


def ring_merge(partial: Partial, *, world: int, rank: int, exchange: Callable[[Partial, int, int, int], Partial],
               merge: Callable[[Partial, Partial], Partial] = rau_merge) -> Partial:
    """Runs this rank's side of the ring: returns the merge of every rank's partial.

    exchange(send, send_to, recv_from, step) sends `send` to rank send_to and returns the
    partial received from rank recv_from (both complete on return); merge(acc, part)
    returns the merged partial without modifying its arguments."""
    acc = partial
    send = partial
    for step, dst, src, _origin in ring_steps(world, rank):
        recv = exchange(send, dst, src, step)
        acc = merge(acc, recv)
        send = recv
    return acc


class DistExchange:
    """Point-to-point exchange of partials through torch.distributed (any backend with
    send/recv: NCCL across GPUs, gloo across CPU processes)."""

    def __init__(self, group=None):
        self.group = group

    def __call__(self, send: Partial, dst: int, src: int, step: int) -> Partial:
        import torch.distributed as dist
        recv = tuple(torch.empty_like(t) for t in send)
        ops = [dist.P2POp(dist.isend, t.contiguous(), dst, self.group) for t in send]
        ops += [dist.P2POp(dist.irecv, t, src, self.group) for t in recv]
        for work in dist.batch_isend_irecv(ops):
            work.wait()
        return recv


def shard_tables(block_table: torch.Tensor, lengths: torch.Tensor, *, world: int, max_kv_len: int,
                 block_size: int) -> Tuple[int, List[torch.Tensor], List[torch.Tensor]]:
    """Splits a paged cache's keys into `world` shards of S tokens (S = max_kv_len / world
    rounded up to whole blocks): shard r holds keys [r S, (r + 1) S) of every sequence.
    Returns S and, per shard, its block-table columns and its per-sequence key counts."""
    per = -(-max_kv_len // world) if world else 0
    S = max(-(-per // block_size) * block_size, block_size)
    cols = S // block_size
    tables, lens = [], []
    for r in range(world):
        t = block_table[:, r * cols:(r + 1) * cols]
        if t.shape[1] < cols:  # past the table's width: columns never read (their keys do not exist)
            pad = torch.full((block_table.shape[0], cols - t.shape[1]), -1, dtype=block_table.dtype,
                             device=block_table.device)
            t = torch.cat([t, pad], dim=1)
        tables.append(t.contiguous())
        lens.append((lengths - r * S).clamp(0, S).contiguous())
    return S, tables, lens


def ring_decode_streams(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_table: torch.Tensor,
                        actual_seq_lengths: torch.Tensor, *, world: int, max_kv_len: int, num_heads: int,
                        num_kv_heads: int = 0, scale: Optional[float] = None, antiquant_scale=None,
                        antiquant_offset=None, sink: Optional[torch.Tensor] = None, num_splits: int = 0,
                        streams: Optional[Sequence[torch.cuda.Stream]] = None) -> List[Partial]:
    """The ring on one GPU: `world` ranks as CUDA streams.  Rank r runs fia_decode over shard r
    (shard_tables) on its stream, then the steps of ring_steps, each receive a device copy
    from the sender's buffer into one of the receiver's two buffers (the step's parity),
    each merge ring_attention_update on the receiver's stream.  Events order the ranks:
    a copy waits until the sender's buffer holds that step's partial, and a rank refills a
    buffer only after the next rank has copied what it held.  Returns every rank's merged
    (out, max, sum) (B, Nq, D) / (B, Nq); the caller's current stream waits for all of them."""
    if world < 1:
        raise ValueError("world must be >= 1")
    B, D = int(q.shape[0]), int(q.shape[-1])
    nkv = num_kv_heads if num_kv_heads else num_heads
    block_size = int(k_cache.shape[2])
    S, tables, lens = shard_tables(block_table, actual_seq_lengths, world=world, max_kv_len=max_kv_len,
                                   block_size=block_size)
    caller = torch.cuda.current_stream()
    # under stream capture the graph's private pool keeps every buffer for the graph's life
    capturing = torch.cuda.is_current_stream_capturing()
    if streams is None:
        streams = [torch.cuda.Stream(device=q.device) for _ in range(world)]
    ws_bytes = fia_decode_workspace_size(B, num_heads, nkv, D, S, block_size, num_splits)

    def new_partial():
        return (torch.empty((B, num_heads, D), dtype=q.dtype, device=q.device),
                torch.empty((B, num_heads), dtype=torch.float32, device=q.device),
                torch.empty((B, num_heads), dtype=torch.float32, device=q.device))

    own, acc, bufs, ready, copied = [], [], [], [], []
    start = torch.cuda.Event()
    start.record(caller)
    for r in range(world):
        with torch.cuda.stream(streams[r]):
            streams[r].wait_event(start)  # the inputs are ready on the caller's stream
            part = new_partial()
            ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
            fia_decode(q, k_cache, v_cache, tables[r], lens[r], max_kv_len=S, num_heads=num_heads,
                       num_kv_heads=nkv, scale=scale, antiquant_scale=antiquant_scale,
                       antiquant_offset=antiquant_offset, sink=sink if r == 0 else None, out=part[0],
                       softmax_max=part[1], softmax_sum=part[2], num_splits=num_splits, workspace=ws)
            ev = torch.cuda.Event()
            ev.record(streams[r])
            own.append(part)
            acc.append(new_partial())
            bufs.append((new_partial(), new_partial()))
            ready.append({0: ev})  # ready[r][s]: rank r's send buffer for step s + 1 holds its partial
            copied.append({})      # copied[r][s]: rank r has copied what it received at step s
    for s in range(1, world):
        for r in range(world):
            src = (r - 1) % world
            nxt = (r + 1) % world
            st = streams[r]
            with torch.cuda.stream(st):
                st.wait_event(ready[src][s - 1])
                if s >= 3:  # buffer s % 2 last held step s - 2's partial, which rank r + 1 copied at s - 1
                    st.wait_event(copied[nxt][s - 1])
                send = own[src] if s == 1 else bufs[src][(s - 1) % 2]
                dst = bufs[r][s % 2]
                for d, x in zip(dst, send):
                    d.copy_(x, non_blocking=True)
                    if not capturing:
                        x.record_stream(st)  # allocated on the sender's stream, read on this one
                ev = torch.cuda.Event()
                ev.record(st)
                copied[r][s] = ev
                ready[r][s] = ev
                prev = own[r] if s == 1 else acc[r]
                ring_attention_update(*prev, *dst, out=acc[r][0], max_out=acc[r][1], sum_out=acc[r][2])
    for r in range(world):
        if world == 1:
            with torch.cuda.stream(streams[r]):
                for d, x in zip(acc[r], own[r]):
                    d.copy_(x, non_blocking=True)
        caller.wait_stream(streams[r])
    # the buffers were allocated on the ranks' streams and are used there until the caller's
    # wait above; tell the caching allocator which streams still use the results
    if not capturing:
        for r in range(world):
            for t in acc[r]:
                t.record_stream(caller)
    return acc


class RingDecodeGraph:
    """One ring step (ring_decode_streams over fixed input tensors) captured in a CUDA graph.

    On one GPU a ring step issues a few hundred operations (W decodes, W (W - 1) copies and
    merges, the events between them); issued from Python they cost more host time than the
    GPU spends on them.  Captured once, a step is one graph launch.  The inputs are read at
    replay time, so new contents of the same tensors give new results; `out` holds every
    rank's (out, max, sum), rewritten by each replay."""

    def __init__(self, q, k_cache, v_cache, block_table, actual_seq_lengths, *, world: int, **kw):
        self.streams = [torch.cuda.Stream(device=q.device) for _ in range(world)]
        args = (q, k_cache, v_cache, block_table, actual_seq_lengths)
        # one eager step first: the library's per-device set-up (device properties, kernel
        # attributes) then happens outside the capture
        ring_decode_streams(*args, world=world, streams=self.streams, **kw)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=torch.cuda.Stream(device=q.device)):
            self.out = ring_decode_streams(*args, world=world, streams=self.streams, **kw)

    def replay(self) -> List[Partial]:
        self.graph.replay()
        return self.out
