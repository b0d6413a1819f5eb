"""Pins for the oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError if
the oracle disagrees with what the operator pages or the mathematics fix:

* library routines on special cases: torch's scaled_dot_product_attention in
  fp64 on the CPU (dense keys, GQA by explicit head repetition, the sink as an
  extra zero-value key whose logit is set through an additive mask, causal
  masks as explicit lower-triangular boolean matrices); scipy's logsumexp for
  the softmax max/sum;
* closed forms: V = ones gives ones; one visible key gives its value row; the
  sink formula with one key; equal scores under a causal mask give 1/(i+1);
* worked examples printed on the pages (stored under tests/golden/);
* invariants: paged layout == contiguous layout bit for bit; sink = -inf ==
  no sink bit for bit; any split of the keys merged by RingAttentionUpdate ==
  unsplit; the literal printed RingAttentionUpdate formula is *not* exact;
* exact fp32 semantics of the int8 antiquant, compared with numpy float32.

tests/test_oracle_mutants.py compiles copies of the oracle with planted
mistakes and checks that every one of them fails at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
from scipy.special import logsumexp

import fia_workloads as W
import oracle as OR

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ references
def sdpa_rows(q, K, V, scale, *, bool_mask=None, add_mask=None):
    """torch SDPA (fp64, CPU) for query rows q (H, Lq, D) over K, V (H, Lk, D)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    mask = None
    if bool_mask is not None:
        mask = torch.from_numpy(np.ascontiguousarray(bool_mask))
    if add_mask is not None:
        mask = t(add_mask)
    o = torch.nn.functional.scaled_dot_product_attention(t(q)[None], t(K)[None], t(V)[None],
                                                         attn_mask=mask, scale=scale)
    return o[0].numpy()


def lse_max_sum(scores):
    """(max, sum of e^{s - max}) along the last axis via scipy's logsumexp."""
    m = np.max(scores, axis=-1)
    return m, np.exp(logsumexp(scores, axis=-1) - m)


def _dense_case(rng, B, Nq, Nkv, D, lengths, dtype=W.BF16):
    """Dense per-batch K/V (B, Nkv, Lmax, D) in storage bits plus the fp32 view."""
    Lmax = max(max(lengths), 1)
    q = W.to_bits(rng.standard_normal((B, Nq, D), dtype=np.float32), dtype)
    k = W.to_bits(rng.standard_normal((B, Nkv, Lmax, D), dtype=np.float32), dtype)
    v = W.to_bits(rng.standard_normal((B, Nkv, Lmax, D), dtype=np.float32), dtype)
    return q, k, v, Lmax


def _code(dtype):
    return OR.BF16 if dtype == W.BF16 else OR.F16


# ------------------------------------------------------------------ decode pins
def pin_decode_matches_sdpa_gqa(O):
    """Decode over a shuffled paged cache equals torch SDPA with K/V heads repeated per group."""
    rng = np.random.default_rng(7)
    for (B, Nq, Nkv, D, lengths, bs, dtype) in [
        (3, 6, 2, 8, [1, 5, 9], 4, W.BF16),
        (2, 4, 4, 16, [17, 3], 8, W.FP16),
        (1, 8, 1, 32, [40], 16, W.BF16),
    ]:
        case = W.make_decode_case(B=B, Nq=Nq, Nkv=Nkv, D=D, block_size=bs, dtype=dtype,
                                  lengths=lengths, seed=int(rng.integers(1 << 30)), scale=0.37)
        out, mx, sm = O.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=Nq, Nkv=Nkv, D=D,
                               scale=case.scale, q_dtype=_code(dtype), kv_dtype=_code(dtype),
                               block_table=case.block_table, block_size=bs)
        q32 = W.bits_to_f32(case.q, dtype).astype(np.float64)
        kc = W.bits_to_f32(case.k_cache, dtype).astype(np.float64)
        vc = W.bits_to_f32(case.v_cache, dtype).astype(np.float64)
        G = Nq // Nkv
        for b in range(B):
            L = int(case.lengths[b])
            blocks = case.block_table[b, :(L + bs - 1) // bs]
            K = np.concatenate([kc[p] for p in blocks], axis=1)[:, :L]   # (Nkv, L, D)
            V = np.concatenate([vc[p] for p in blocks], axis=1)[:, :L]
            Kr, Vr = np.repeat(K, G, axis=0), np.repeat(V, G, axis=0)    # (Nq, L, D)
            ref = sdpa_rows(q32[b][:, None, :], Kr, Vr, case.scale)[:, 0, :]
            m_ref, s_ref = lse_max_sum(case.scale * np.einsum("hd,hld->hl", q32[b], Kr))
            rows = slice(b * Nq, (b + 1) * Nq)
            np.testing.assert_allclose(out[rows], ref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(mx[rows], m_ref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(sm[rows], s_ref, rtol=1e-12, atol=1e-12)


def pin_decode_sink_matches_sdpa(O):
    """The sink equals one more key with value row 0 whose logit is the sink (additive mask)."""
    rng = np.random.default_rng(11)
    B, Nq, Nkv, D, L = 2, 4, 2, 8, 6
    q, k, v, _ = _dense_case(rng, B, Nq, Nkv, D, [L, L])
    sink = rng.standard_normal(Nq).astype(np.float32) * 3
    scale = 0.5
    out, mx, sm = O.decode(q, k, v, [L, L], Nq=Nq, Nkv=Nkv, D=D, scale=scale, q_dtype=OR.BF16,
                           kv_dtype=OR.BF16, kv_rows=L, sink=sink)
    q32 = W.bits_to_f32(q, W.BF16).astype(np.float64)
    K = np.repeat(W.bits_to_f32(k, W.BF16).astype(np.float64), Nq // Nkv, axis=1)
    V = np.repeat(W.bits_to_f32(v, W.BF16).astype(np.float64), Nq // Nkv, axis=1)
    for b in range(B):
        Ke = np.concatenate([K[b], np.zeros((Nq, 1, D))], axis=1)       # key L+1: all zeros
        Ve = np.concatenate([V[b], np.zeros((Nq, 1, D))], axis=1)
        add = np.zeros((Nq, 1, L + 1))
        add[:, 0, L] = sink                                             # its logit := sink
        ref = sdpa_rows(q32[b][:, None, :], Ke, Ve, scale, add_mask=add)[:, 0, :]
        s = scale * np.einsum("hd,hld->hl", q32[b], K[b])
        m_ref, s_ref = lse_max_sum(np.concatenate([s, sink[:, None].astype(np.float64)], axis=1))
        rows = slice(b * Nq, (b + 1) * Nq)
        np.testing.assert_allclose(out[rows], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(mx[rows], m_ref, rtol=1e-12, atol=0)
        np.testing.assert_allclose(sm[rows], s_ref, rtol=1e-12, atol=0)


def pin_v_ones_gives_ones(O):
    """Softmax rows sum to one: with V = 1 every output element is 1."""
    rng = np.random.default_rng(3)
    B, Nq, Nkv, D = 2, 4, 2, 16
    q, k, _, Lmax = _dense_case(rng, B, Nq, Nkv, D, [13, 29])
    v = np.full_like(k, W.to_bf16_bits(np.ones(1, np.float32))[0])
    out, _, _ = O.decode(q, k, v, [13, 29], Nq=Nq, Nkv=Nkv, D=D, scale=0.25, q_dtype=OR.BF16,
                         kv_dtype=OR.BF16, kv_rows=Lmax)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-12)


def pin_ifa_v3_worked_example(O):
    """aclnnIncreFlashAttentionV3 example program: all-ones fp16 inputs, scale 1/sqrt(16)."""
    g = golden("ifa_v3_example.json")
    B, N, D, S = g["batch"], g["num_heads"], g["head_dims"], g["seq_len_kv"]
    one = W.to_f16_bits(np.ones(1, np.float32))[0]
    q = np.full((B, N, D), one, np.uint16)
    k = np.full((B, g["num_kv_heads"], S, D), one, np.uint16)
    out, mx, sm = O.decode(q, k, k, [S] * B, Nq=N, Nkv=g["num_kv_heads"], D=D,
                           scale=1.0 / math.sqrt(D), q_dtype=OR.F16, kv_dtype=OR.F16, kv_rows=S)
    assert np.all(out == g["expected_out_value"])
    assert np.all(mx == g["expected_softmax_max"])
    assert np.all(sm == g["expected_softmax_sum"])


def pin_single_key_returns_its_value(O):
    """One visible key: out = v_0 exactly, max = its logit, sum = 1 (fp16 specials included)."""
    D = 8
    vals = np.array([1.0, -2.5, 65504.0, 6.0e-8, -0.0, 3.140625, 1e-5, -7.75], np.float32)
    for dtype, code in [(W.FP16, OR.F16), (W.BF16, OR.BF16)]:
        v = W.to_bits(vals, dtype).reshape(1, 1, 1, D)
        k = W.to_bits(np.array([0.5, 1, -1, 2, 0, 0.25, 4, -0.5], np.float32), dtype).reshape(1, 1, 1, D)
        q = W.to_bits(np.array([1, 2, 0.5, -1, 3, 4, 0.125, 2], np.float32), dtype).reshape(1, 1, D)
        out, mx, sm = O.decode(q, k, v, [1], Nq=1, Nkv=1, D=D, scale=0.5, q_dtype=code, kv_dtype=code,
                               kv_rows=1)
        v64 = W.bits_to_f32(v, dtype).astype(np.float64).reshape(D)
        assert np.array_equal(out[0], v64)
        logit = 0.5 * float(np.dot(W.bits_to_f32(q, dtype).astype(np.float64).reshape(D),
                                   W.bits_to_f32(k, dtype).astype(np.float64).reshape(D)))
        assert mx[0] == logit and sm[0] == 1.0


def pin_paged_equals_contiguous(O):
    """Reading through a shuffled block table gives the contiguous layout's result bit for bit."""
    rng = np.random.default_rng(5)
    B, Nq, Nkv, D, bs = 3, 4, 2, 16, 4
    lengths = [9, 1, 16]
    q, k, v, Lmax = _dense_case(rng, B, Nq, Nkv, D, lengths)
    nblk = [(L + bs - 1) // bs for L in lengths]
    perm = rng.permutation(sum(nblk) + 2)                     # two spare blocks
    table = np.full((B, max(nblk) + 1), -1, np.int32)
    kp = np.zeros((len(perm), Nkv, bs, D), np.uint16)
    vp = np.zeros_like(kp)
    nxt = 0
    for b in range(B):
        for i in range(nblk[b]):
            p = perm[nxt]
            nxt += 1
            table[b, i] = p
            rows = slice(i * bs, min((i + 1) * bs, Lmax))
            kp[p, :, :rows.stop - rows.start] = k[b, :, rows]
            vp[p, :, :rows.stop - rows.start] = v[b, :, rows]
    a = O.decode(q, k, v, lengths, Nq=Nq, Nkv=Nkv, D=D, scale=0.3, q_dtype=OR.BF16, kv_dtype=OR.BF16,
                 kv_rows=Lmax)
    p_ = O.decode(q, kp, vp, lengths, Nq=Nq, Nkv=Nkv, D=D, scale=0.3, q_dtype=OR.BF16,
                  kv_dtype=OR.BF16, block_table=table, block_size=bs)
    for x, y in zip(a, p_):
        assert np.array_equal(x, y)


def pin_sink_minus_inf_is_no_sink(O):
    rng = np.random.default_rng(9)
    q, k, v, L = _dense_case(rng, 2, 4, 2, 8, [7, 7])
    kw = dict(Nq=4, Nkv=2, D=8, scale=0.4, q_dtype=OR.BF16, kv_dtype=OR.BF16, kv_rows=L)
    a = O.decode(q, k, v, [7, 5], **kw)
    b = O.decode(q, k, v, [7, 5], sink=np.full(4, -np.inf, np.float32), **kw)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def pin_sink_single_key_closed_form(O):
    """One key with logit s and a sink c: out = v e^s / (e^s + e^c), max = max(s, c)."""
    D = 4
    q = W.to_bf16_bits(np.array([1.0, 2.0, -1.0, 0.5], np.float32)).reshape(1, 1, D)
    k = W.to_bf16_bits(np.array([0.5, 0.25, 1.0, 2.0], np.float32)).reshape(1, 1, 1, D)
    v = W.to_bf16_bits(np.array([3.0, -1.0, 0.5, 8.0], np.float32)).reshape(1, 1, 1, D)
    s = 1.0 * (0.5 + 0.5 - 1.0 + 1.0)
    for c in [-3.0, 0.0, 0.75, 2.5]:
        out, mx, sm = O.decode(q, k, v, [1], Nq=1, Nkv=1, D=D, scale=1.0, q_dtype=OR.BF16,
                               kv_dtype=OR.BF16, kv_rows=1, sink=np.array([c], np.float32))
        ref = np.array([3.0, -1.0, 0.5, 8.0]) * math.exp(s) / (math.exp(s) + math.exp(c))
        np.testing.assert_allclose(out[0], ref, rtol=1e-14, atol=0)
        assert mx[0] == max(s, c)
        np.testing.assert_allclose(sm[0], (math.exp(s) + math.exp(c)) / math.exp(max(s, c)), rtol=1e-14)


def pin_sink_large_drives_out_to_zero(O):
    rng = np.random.default_rng(13)
    q, k, v, L = _dense_case(rng, 1, 2, 1, 8, [5])
    out, mx, sm = O.decode(q, k, v, [5], Nq=2, Nkv=1, D=8, scale=0.3, q_dtype=OR.BF16,
                           kv_dtype=OR.BF16, kv_rows=L, sink=np.array([1000.0, 1000.0], np.float32))
    assert np.all(np.abs(out) < 1e-300) and np.all(mx == 1000.0) and np.all(sm == 1.0)


def pin_empty_kv(O):
    """No visible key: out 0, max -inf, sum 0; with a sink: out 0, max = sink, sum 1."""
    rng = np.random.default_rng(17)
    q, k, v, L = _dense_case(rng, 2, 2, 1, 8, [4, 0])
    out, mx, sm = O.decode(q, k, v, [4, 0], Nq=2, Nkv=1, D=8, scale=0.3, q_dtype=OR.BF16,
                           kv_dtype=OR.BF16, kv_rows=L)
    assert np.all(out[2:] == 0) and np.all(mx[2:] == -np.inf) and np.all(sm[2:] == 0)
    out, mx, sm = O.decode(q, k, v, [4, 0], Nq=2, Nkv=1, D=8, scale=0.3, q_dtype=OR.BF16,
                           kv_dtype=OR.BF16, kv_rows=L, sink=np.array([0.5, -2.0], np.float32))
    assert np.all(out[2:] == 0) and np.array_equal(mx[2:], [0.5, -2.0]) and np.all(sm[2:] == 1)


def pin_decode_mask_matches_sdpa(O):
    """attenMask (B, 1, 1, S): a nonzero byte removes the key; equals torch SDPA with the
    boolean mask (True = attend) over the paged keys gathered by the block table."""
    rng = np.random.default_rng(23)
    B, Nq, Nkv, D, bs = 3, 4, 2, 16, 8
    lengths = [13, 30, 7]
    case = W.make_decode_case(B=B, Nq=Nq, Nkv=Nkv, D=D, block_size=bs, lengths=lengths, seed=23, scale=0.41)
    S = 32                                              # mask row longer than every length
    mask = rng.random((B, S)) < 0.35
    mask[2, :7] = True                                  # batch 2: every key masked
    out, mx, sm = O.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=Nq, Nkv=Nkv, D=D,
                           scale=case.scale, q_dtype=OR.BF16, kv_dtype=OR.BF16,
                           block_table=case.block_table, block_size=bs, mask=mask.astype(np.uint8))
    q32 = W.bits_to_f32(case.q, W.BF16).astype(np.float64)
    kc = W.bits_to_f32(case.k_cache, W.BF16).astype(np.float64)
    vc = W.bits_to_f32(case.v_cache, W.BF16).astype(np.float64)
    G = Nq // Nkv
    for b in range(2):
        L = lengths[b]
        blocks = case.block_table[b, :(L + bs - 1) // bs]
        K = np.repeat(np.concatenate([kc[p] for p in blocks], axis=1)[:, :L], G, axis=0)
        V = np.repeat(np.concatenate([vc[p] for p in blocks], axis=1)[:, :L], G, axis=0)
        keep = np.broadcast_to(~mask[b, :L], (Nq, 1, L))
        ref = sdpa_rows(q32[b][:, None, :], K, V, case.scale, bool_mask=keep)[:, 0, :]
        sc = case.scale * np.einsum("hd,hld->hl", q32[b], K)[:, ~mask[b, :L]]
        m_ref, s_ref = lse_max_sum(sc)
        rows = slice(b * Nq, (b + 1) * Nq)
        np.testing.assert_allclose(out[rows], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(mx[rows], m_ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(sm[rows], s_ref, rtol=1e-12, atol=1e-12)
    rows = slice(2 * Nq, 3 * Nq)                        # fully masked: the empty-row values
    assert np.all(out[rows] == 0) and np.all(mx[rows] == -np.inf) and np.all(sm[rows] == 0)
    # an all-zero mask is no mask, bit for bit; bool, int8 and uint8 masks agree
    ref = O.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=Nq, Nkv=Nkv, D=D, scale=case.scale,
                   q_dtype=OR.BF16, kv_dtype=OR.BF16, block_table=case.block_table, block_size=bs)
    zero = O.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=Nq, Nkv=Nkv, D=D, scale=case.scale,
                    q_dtype=OR.BF16, kv_dtype=OR.BF16, block_table=case.block_table, block_size=bs,
                    mask=np.zeros((B, S), np.int8))
    assert all(np.array_equal(x, y) for x, y in zip(ref, zero))
    asb = O.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=Nq, Nkv=Nkv, D=D, scale=case.scale,
                   q_dtype=OR.BF16, kv_dtype=OR.BF16, block_table=case.block_table, block_size=bs, mask=mask)
    assert all(np.array_equal(x, y) for x, y in zip(asb, (out, mx, sm)))


def pin_decode_band_is_prefill_band_of_one_query(O):
    """Decode with a band (pre, next) over a shuffled paged cache equals the prefill oracle's
    band (pinned against SDPA with triu/tril masks) for one query per sequence over the
    gathered keys, and an attenMask that masks the keys outside the window."""
    B, Nq, Nkv, D, bs = 3, 4, 2, 16, 8
    lengths = [30, 5, 17]
    case = W.make_decode_case(B=B, Nq=Nq, Nkv=Nkv, D=D, block_size=bs, lengths=lengths, seed=37, scale=0.45)
    kc = case.k_cache.transpose(0, 2, 1, 3)   # (blocks, bs, Nkv, D)
    vc = case.v_cache.transpose(0, 2, 1, 3)
    k = np.concatenate([np.concatenate([kc[p] for p in case.block_table[b, :(L + bs - 1) // bs]])[:L]
                        for b, L in enumerate(lengths)])
    v = np.concatenate([np.concatenate([vc[p] for p in case.block_table[b, :(L + bs - 1) // bs]])[:L]
                        for b, L in enumerate(lengths)])
    cu_q = np.arange(B + 1)
    cu_kv = np.concatenate([[0], np.cumsum(lengths)])
    for pre, nxt in [(7, 0), (0, 0), (3, -1), (100, 0), (12, -10)]:
        dec = O.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=Nq, Nkv=Nkv, D=D, scale=case.scale,
                       q_dtype=OR.BF16, kv_dtype=OR.BF16, block_table=case.block_table, block_size=bs,
                       band=(pre, nxt))
        pf = O.prefill(case.q, k, v, cu_q, cu_kv, Nq=Nq, Nkv=Nkv, D=D, scale=case.scale, dtype=OR.BF16,
                       band=(pre, nxt))
        for x, y in zip(dec, pf):
            np.testing.assert_allclose(x, y, rtol=1e-13, atol=1e-13)
        mask = np.ones((B, 32), np.uint8)
        for b, L in enumerate(lengths):
            mask[b, max(0, L - 1 - pre):max(0, min(L, L + nxt))] = 0
        msk = O.decode(case.q, case.k_cache, case.v_cache, case.lengths, Nq=Nq, Nkv=Nkv, D=D, scale=case.scale,
                       q_dtype=OR.BF16, kv_dtype=OR.BF16, block_table=case.block_table, block_size=bs, mask=mask)
        assert all(np.array_equal(x, y) for x, y in zip(dec, msk))


def pin_decode_query_positions(O):
    """s query positions per batch (the last s of each sequence): equal to the prefill oracle
    with Lq = s over the gathered keys (causal, and with a band), and to torch SDPA under a
    mask built with numpy's tril (k = L - s); a position before the first key gets the empty
    row."""
    rng = np.random.default_rng(41)
    B, Nq, Nkv, D, bs, s = 3, 4, 2, 16, 8, 3
    lengths = [30, 2, 17]
    case = W.make_decode_case(B=B, Nq=Nq, Nkv=Nkv, D=D, block_size=bs, lengths=lengths, seed=41, scale=0.4)
    q = W.to_bits(rng.standard_normal((B, s, Nq, D), dtype=np.float32), W.BF16)
    kc = case.k_cache.transpose(0, 2, 1, 3)
    vc = case.v_cache.transpose(0, 2, 1, 3)
    k = np.concatenate([np.concatenate([kc[p] for p in case.block_table[b, :(L + bs - 1) // bs]])[:L]
                        for b, L in enumerate(lengths)])
    v = np.concatenate([np.concatenate([vc[p] for p in case.block_table[b, :(L + bs - 1) // bs]])[:L]
                        for b, L in enumerate(lengths)])
    cu_q = np.arange(B + 1) * s
    cu_kv = np.concatenate([[0], np.cumsum(lengths)])
    kw = dict(Nq=Nq, Nkv=Nkv, D=D, scale=case.scale)
    for band in [None, (4, 0), (1, -1)]:
        dec = O.decode(q, case.k_cache, case.v_cache, case.lengths, q_dtype=OR.BF16, kv_dtype=OR.BF16,
                       block_table=case.block_table, block_size=bs, band=band, q_len=s, **kw)
        pf = O.prefill(q.reshape(B * s, Nq, D), k, v, cu_q, cu_kv, dtype=OR.BF16, causal=True, band=band, **kw)
        for x, y in zip(dec, pf):
            np.testing.assert_allclose(x, y, rtol=1e-13, atol=1e-13)
    out, mx, sm = O.decode(q, case.k_cache, case.v_cache, case.lengths, q_dtype=OR.BF16, kv_dtype=OR.BF16,
                           block_table=case.block_table, block_size=bs, q_len=s, **kw)
    qf = W.bits_to_f32(q, W.BF16).astype(np.float64)
    kf = np.repeat(W.bits_to_f32(k, W.BF16).astype(np.float64), Nq // Nkv, axis=1)
    vf = np.repeat(W.bits_to_f32(v, W.BF16).astype(np.float64), Nq // Nkv, axis=1)
    for b, L in enumerate(lengths):
        allowed = np.tril(np.ones((s, L), bool), k=L - s)
        has = allowed.any(axis=1)
        rows = (np.arange(s)[:, None] + b * s) * Nq + np.arange(Nq)[None, :]    # (s, Nq)
        K = kf[cu_kv[b]:cu_kv[b + 1]].transpose(1, 0, 2)
        V = vf[cu_kv[b]:cu_kv[b + 1]].transpose(1, 0, 2)
        Q = qf[b][has].transpose(1, 0, 2)                                        # (Nq, s', D)
        ref = sdpa_rows(Q, K, V, case.scale, bool_mask=np.broadcast_to(allowed[has], (Nq,) + allowed[has].shape))
        np.testing.assert_allclose(out[rows[has].T], ref, rtol=1e-12, atol=1e-12)
        e = rows[~has]
        assert np.all(out[e] == 0) and np.all(mx[e] == -np.inf) and np.all(sm[e] == 0)
    one = O.decode(case.q, case.k_cache, case.v_cache, case.lengths, q_dtype=OR.BF16, kv_dtype=OR.BF16,
                   block_table=case.block_table, block_size=bs, q_len=1, **kw)
    ref = O.decode(case.q, case.k_cache, case.v_cache, case.lengths, q_dtype=OR.BF16, kv_dtype=OR.BF16,
                   block_table=case.block_table, block_size=bs, **kw)
    assert all(np.array_equal(x, y) for x, y in zip(one, ref))


# ------------------------------------------------------------------ post-quant output
def pin_post_quant_closed_forms(O):
    """Ties go to the even integer, values past the int8 range saturate, the offset is added."""
    x = np.array([[0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 0.49, 126.5, 127.5, 128.0, 1e6,
                   -127.5, -128.5, -129.0, -1e6, 3.2]])
    y, code = O.post_quant(x, [1.0])
    assert np.array_equal(y, x)
    assert code.tolist() == [[0, 2, 2, 0, -2, -2, 0, 126, 127, 127, 127, -128, -128, -128, -128, 3]]
    _, code = O.post_quant(np.array([[1.0, -1.0, 0.25]]), [2.0], [0.5])   # 2.5, -1.5, 1.0
    assert code.tolist() == [[2, -2, 1]]


def pin_post_quant_matches_numpy(O):
    """Per-tensor and per-channel (channel h * D + d of an (N, D) row) against numpy's rint
    (ties to even) and clip."""
    rng = np.random.default_rng(29)
    R, N, D = 5, 3, 8
    x = rng.standard_normal((R, N, D)) * 40
    s_c = rng.uniform(0.5, 3.0, N * D).astype(np.float32)
    o_c = rng.uniform(-20, 20, N * D).astype(np.float32)
    for s2, o2 in [(s_c[:1], None), (s_c[:1], o_c[:1]), (s_c, None), (s_c, o_c)]:
        y, code = O.post_quant(x, s2, o2)
        s_b = np.broadcast_to(s2.astype(np.float64), (N * D,)).reshape(N, D)
        o_b = 0.0 if o2 is None else np.broadcast_to(o2.astype(np.float64), (N * D,)).reshape(N, D)
        y_ref = x * s_b + o_b
        np.testing.assert_allclose(y, y_ref, rtol=1e-15, atol=0)
        assert np.array_equal(code, np.clip(np.rint(y_ref), -128, 127).astype(np.int8))


# ------------------------------------------------------------------ int8 antiquant
def pin_dequant_fp32_semantics(O):
    """(x - offset) * scale as two fp32 round-to-nearest operations, for all 256 codes."""
    rng = np.random.default_rng(19)
    codes = np.arange(-128, 128, dtype=np.int32)
    offs = np.concatenate([[0.0, 1.5, -2.0], rng.uniform(-2, 2, 5)]).astype(np.float32)
    scs = np.concatenate([[1.0, 0.0078125], rng.uniform(0.005, 0.02, 6)]).astype(np.float32)
    for off, sc in zip(offs, scs):
        ref = (codes.astype(np.float32) - np.float32(off)) * np.float32(sc)   # numpy fp32 ops
        got = np.array([O.dequant_i8(int(x), float(off), float(sc)) for x in codes], np.float32)
        assert np.array_equal(ref.view(np.uint32), got.view(np.uint32))
    assert O.dequant_i8(-77, 0.0, 1.0) == -77.0


def pin_int8_decode_uses_k_and_v_params(O):
    """One visible key: out = dequantised V row (index 1 of the params), logit from index 0."""
    rng = np.random.default_rng(23)
    Nkv, D, G = 2, 8, 2
    kc = rng.integers(-127, 128, size=(1, Nkv, 1, D)).astype(np.int8)
    vc = rng.integers(-127, 128, size=(1, Nkv, 1, D)).astype(np.int8)
    sc = rng.uniform(0.005, 0.02, size=(2, Nkv, D)).astype(np.float32)
    off = rng.uniform(-2, 2, size=(2, Nkv, D)).astype(np.float32)
    q = W.to_bf16_bits(rng.standard_normal((1, Nkv * G, D), dtype=np.float32))
    out, mx, sm = O.decode(q, kc, vc, [1], Nq=Nkv * G, Nkv=Nkv, D=D, scale=0.7, q_dtype=OR.BF16,
                           kv_dtype=OR.I8, kv_rows=1, aq_scale=sc, aq_offset=off)
    q64 = W.bits_to_f32(q, W.BF16).astype(np.float64)[0]
    for h in range(Nkv * G):
        hk = h // G
        khat = ((kc[0, hk, 0].astype(np.float32) - off[0, hk]) * sc[0, hk]).astype(np.float64)
        vhat = ((vc[0, hk, 0].astype(np.float32) - off[1, hk]) * sc[1, hk]).astype(np.float64)
        assert np.array_equal(out[h], vhat)
        np.testing.assert_allclose(mx[h], 0.7 * np.dot(q64[h], khat), rtol=1e-13)
        assert sm[h] == 1.0


def pin_dequant_array_matches_numpy(O):
    """The array form of the antiquant step equals numpy fp32 (x - offset) * scale."""
    rng = np.random.default_rng(43)
    codes = np.tile(np.arange(-128, 128, dtype=np.int8), 9)
    off = rng.uniform(-2, 2, codes.size).astype(np.float32)
    sc = rng.uniform(0.005, 0.02, codes.size).astype(np.float32)
    ref = (codes.astype(np.float32) - off) * sc
    assert np.array_equal(O.dequant_i8_array(codes, off, sc).view(np.uint32), ref.view(np.uint32))


def pin_gather_rows_inverts_a_scatter(O):
    """Scatter a contiguous K into a shuffled pool by hand; the oracle's gather gives it back."""
    rng = np.random.default_rng(47)
    Nkv, D, bs, L = 3, 8, 16, 53
    k = rng.integers(0, 1 << 16, size=(Nkv, L, D)).astype(np.uint16)
    nblk = (L + bs - 1) // bs
    perm = rng.permutation(nblk + 4)
    pool = rng.integers(0, 1 << 16, size=(nblk + 4, Nkv, bs, D)).astype(np.uint16)
    table = np.full((2, nblk + 2), -1, np.int32)
    table[1, :nblk] = perm[:nblk]
    for t in range(L):
        pool[perm[t // bs], :, t % bs] = k[:, t]
    for hk in range(Nkv):
        assert np.array_equal(O.gather_rows(pool, table, 1, hk, L, bs), k[hk])


# ------------------------------------------------------------------ split + RingAttentionUpdate
def _row_partials(O, q, k, v, L, lo, hi, D, sink=None):
    """Decode of one row over keys [lo, hi) of a contiguous cache (1, 1, L, D)."""
    out, mx, sm = O.decode(q, k[:, :, lo:hi], v[:, :, lo:hi], [hi - lo], Nq=1, Nkv=1, D=D, scale=0.6,
                           q_dtype=OR.BF16, kv_dtype=OR.BF16, kv_rows=hi - lo, sink=sink)
    return out.reshape(1, 1, D), mx.reshape(1, 1), sm.reshape(1, 1)


def pin_split_then_rau_equals_unsplit(O):
    """Split the keys anywhere (2 parts, and 32 parts), merge by RingAttentionUpdate: unsplit result."""
    rng = np.random.default_rng(29)
    D, L = 8, 64
    q, k, v, _ = _dense_case(rng, 1, 1, 1, D, [L])
    full = _row_partials(O, q, k, v, L, 0, L, D)
    for cut in range(0, L + 1):
        a = _row_partials(O, q, k, v, L, 0, cut, D)
        b = _row_partials(O, q, k, v, L, cut, L, D)
        m = O.rau(*a, *b)
        for x, y in zip(m, full):
            np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-14)
    acc = _row_partials(O, q, k, v, L, 0, 2, D)
    for j in range(1, 32):
        acc = O.rau(*acc, *_row_partials(O, q, k, v, L, 2 * j, 2 * j + 2, D))
    for x, y in zip(acc, full):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-14)
    # a sink given to exactly one chunk enters once
    sink = np.array([0.9], np.float32)
    fs = _row_partials(O, q, k, v, L, 0, L, D, sink=sink)
    m = O.rau(*_row_partials(O, q, k, v, L, 0, 20, D, sink=sink), *_row_partials(O, q, k, v, L, 20, L, D))
    for x, y in zip(m, fs):
        np.testing.assert_allclose(x, y, rtol=1e-12, atol=1e-14)


def pin_rau_literal_formula_is_not_exact(O):
    """A 2-key part merged with a 1-key part: the printed formula (no sum weights) misses the
    unsplit result, the sum-weighted reading hits it."""
    D = 2
    q = W.to_bf16_bits(np.array([1.0, 0.0], np.float32)).reshape(1, 1, D)
    k = W.to_bf16_bits(np.array([[0.0, 0], [0.0, 0], [0.0, 0]], np.float32)).reshape(1, 1, 3, D)
    v = W.to_bf16_bits(np.array([[1.0, 0], [1.0, 0], [4.0, 0]], np.float32)).reshape(1, 1, 3, D)
    full = _row_partials(O, q, k, v, 3, 0, 3, D)
    a = _row_partials(O, q, k, v, 3, 0, 2, D)
    b = _row_partials(O, q, k, v, 3, 2, 3, D)
    (po, pm, ps), (co, cm, cs) = a, b
    m = np.maximum(pm, cm)
    lit_sum = ps * np.exp(pm - m) + np.exp(cm - m)
    lit_out = po * np.exp(pm - m)[..., None] / lit_sum[..., None] + co * np.exp(cm - m)[..., None] / lit_sum[..., None]
    assert abs(lit_out[0, 0, 0] - full[0][0, 0, 0]) > 0.1       # printed formula: 5/3 vs 2
    got = O.rau(*a, *b)
    np.testing.assert_allclose(got[0], full[0], rtol=1e-14)
    np.testing.assert_allclose(full[0][0, 0, 0], 2.0, rtol=1e-14)  # (1 + 1 + 4) / 3


def pin_rau_minus_inf_side(O):
    """A partial with no keys (max -inf, sum 0) leaves the other side unchanged."""
    po = np.array([[[0.25, -1.0]]])
    got = O.rau(po, [[1.5]], [[2.0]], np.zeros((1, 1, 2)), [[-np.inf]], [[0.0]])
    assert np.array_equal(got[0], po) and got[1][0, 0] == 1.5 and got[2][0, 0] == 2.0
    got = O.rau(np.zeros((1, 1, 2)), [[-np.inf]], [[0.0]], np.zeros((1, 1, 2)), [[-np.inf]], [[0.0]])
    assert np.all(got[0] == 0) and got[1][0, 0] == -np.inf and got[2][0, 0] == 0


# ------------------------------------------------------------------ prefill pins
def pin_prefill_matches_sdpa_causal(O):
    """TND prefill equals torch SDPA per sequence with an explicit rightDownCausal mask."""
    rng = np.random.default_rng(31)
    for lengths_q, lengths_kv, Nq, Nkv, D, causal in [
        ([5, 1, 9], None, 4, 2, 8, True),
        ([3, 0, 4], [6, 2, 4], 2, 1, 16, True),    # Lq < Lkv: rightDown offset; an empty sequence
        ([4, 7], None, 2, 2, 8, False),
    ]:
        case = W.make_prefill_case(Nq=Nq, Nkv=Nkv, D=D, lengths=lengths_q, lengths_kv=lengths_kv,
                                   scale=0.45, seed=int(rng.integers(1 << 30)))
        out, mx, sm = O.prefill(case.q, case.k, case.v, case.cu_q, case.cu_kv, Nq=Nq, Nkv=Nkv, D=D,
                                scale=case.scale, causal=causal, dtype=OR.BF16)
        out = out.reshape(case.T, Nq, D)
        mx, sm = mx.reshape(case.T, Nq), sm.reshape(case.T, Nq)
        q32 = W.bits_to_f32(case.q, W.BF16).astype(np.float64)
        k32 = W.bits_to_f32(case.k, W.BF16).astype(np.float64)
        v32 = W.bits_to_f32(case.v, W.BF16).astype(np.float64)
        for b in range(case.B):
            q0, q1 = case.cu_q[b], case.cu_q[b + 1]
            k0, k1 = case.cu_kv[b], case.cu_kv[b + 1]
            Lq, Lk = q1 - q0, k1 - k0
            if Lq == 0 or Lk == 0:
                continue
            Q = q32[q0:q1].transpose(1, 0, 2)                                   # (Nq, Lq, D)
            K = np.repeat(k32[k0:k1].transpose(1, 0, 2), Nq // Nkv, axis=0)
            V = np.repeat(v32[k0:k1].transpose(1, 0, 2), Nq // Nkv, axis=0)
            mask = np.tril(np.ones((Lq, Lk), bool), k=Lk - Lq) if causal else np.ones((Lq, Lk), bool)
            ref = sdpa_rows(Q, K, V, case.scale, bool_mask=mask).transpose(1, 0, 2)
            s = case.scale * np.einsum("hid,hjd->hij", Q, K)
            s = np.where(mask[None], s, -np.inf)
            m_ref, s_ref = lse_max_sum(s)
            np.testing.assert_allclose(out[q0:q1], ref, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(mx[q0:q1], m_ref.T, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(sm[q0:q1], s_ref.T, rtol=1e-12, atol=1e-12)


def pin_prefill_band_matches_sdpa(O):
    """sparseMode 4: the band i + d - pre <= j <= i + d + next (d = Lkv - Lq) equals torch SDPA
    under a boolean mask built with numpy's triu/tril (k = d - pre and d + next); rows with
    no key in the band give the empty-row values; band(huge, 0) is the causal mode and
    band(huge, huge) no mask, bit for bit."""
    rng = np.random.default_rng(31)
    Nq, Nkv, D = 4, 2, 16
    lq, lkv = [9, 1, 14, 6], [9, 5, 20, 3]          # Lq = Lkv, Lq < Lkv and Lq > Lkv
    cu_q = np.concatenate([[0], np.cumsum(lq)])
    cu_kv = np.concatenate([[0], np.cumsum(lkv)])
    T, Tkv = int(cu_q[-1]), int(cu_kv[-1])
    q = W.to_bits(rng.standard_normal((T, Nq, D), dtype=np.float32), W.BF16)
    k = W.to_bits(rng.standard_normal((Tkv, Nkv, D), dtype=np.float32), W.BF16)
    v = W.to_bits(rng.standard_normal((Tkv, Nkv, D), dtype=np.float32), W.BF16)
    f = lambda a: W.bits_to_f32(a, W.BF16).astype(np.float64)
    qf, kf, vf = f(q), np.repeat(f(k), Nq // Nkv, axis=1), np.repeat(f(v), Nq // Nkv, axis=1)
    scale = 0.3
    kw = dict(Nq=Nq, Nkv=Nkv, D=D, scale=scale, dtype=OR.BF16)
    for pre, nxt in [(3, 0), (2, 1), (0, 0), (4, -1), (-1, 2), (1000, 5)]:
        out, mx, sm = O.prefill(q, k, v, cu_q, cu_kv, band=(pre, nxt), **kw)
        for b in range(len(lq)):
            Lq, Lkv = lq[b], lkv[b]
            d = Lkv - Lq
            ones = np.ones((Lq, Lkv), bool)
            allowed = np.triu(ones, k=d - pre) & np.tril(ones, k=d + nxt)
            Q = qf[cu_q[b]:cu_q[b + 1]].transpose(1, 0, 2)
            K = kf[cu_kv[b]:cu_kv[b + 1]].transpose(1, 0, 2)
            V = vf[cu_kv[b]:cu_kv[b + 1]].transpose(1, 0, 2)
            rows = np.arange(cu_q[b] * Nq, cu_q[b + 1] * Nq).reshape(Lq, Nq).T     # (Nq, Lq)
            has = allowed.any(axis=1)
            if has.any():
                ref = sdpa_rows(Q[:, has], K, V, scale, bool_mask=np.broadcast_to(allowed[has], (Nq,) + allowed[has].shape))
                np.testing.assert_allclose(out[rows[:, has]], ref, rtol=1e-12, atol=1e-12)
                s = scale * np.einsum("hid,hjd->hij", Q[:, has], K)
                s = np.where(allowed[has][None], s, -np.inf)
                m_ref, s_ref = lse_max_sum(s)
                np.testing.assert_allclose(mx[rows[:, has]], m_ref, rtol=1e-12, atol=1e-12)
                np.testing.assert_allclose(sm[rows[:, has]], s_ref, rtol=1e-12, atol=1e-12)
            e = rows[:, ~has]
            assert np.all(out[e] == 0) and np.all(mx[e] == -np.inf) and np.all(sm[e] == 0)
    big = 1 << 40
    causal = O.prefill(q, k, v, cu_q, cu_kv, causal=True, **kw)
    assert all(np.array_equal(x, y) for x, y in zip(causal, O.prefill(q, k, v, cu_q, cu_kv, band=(big, 0), **kw)))
    full = O.prefill(q, k, v, cu_q, cu_kv, causal=False, **kw)
    assert all(np.array_equal(x, y) for x, y in zip(full, O.prefill(q, k, v, cu_q, cu_kv, band=(big, big), **kw)))


def pin_prefill_causal_counts(O):
    """Equal scores under the causal mask: query i averages exactly keys 0..i."""
    L, D = 7, 8
    q = np.zeros((L, 1, D), np.float64)
    k = np.zeros((L, 1, D), np.float64)
    v = np.zeros((L, 1, D), np.float64)
    for j in range(L):
        v[j, 0, j] = 1.0                       # value j = unit vector e_j
    cu = np.array([0, L], np.int64)
    out, mx, sm = O.prefill(q, k, v, cu, cu, Nq=1, Nkv=1, D=D, scale=1.0, causal=True)
    for i in range(L):
        ref = np.zeros(D)
        ref[:i + 1] = 1.0 / (i + 1)
        np.testing.assert_allclose(out[i], ref, rtol=1e-15, atol=0)
        assert sm[i] == i + 1 and mx[i] == 0.0


def pin_prefill_rows_without_keys(O):
    """rightDownCausal with Lq > Lkv leaves the first Lq - Lkv rows without keys."""
    rng = np.random.default_rng(37)
    case = W.make_prefill_case(Nq=2, Nkv=1, D=8, lengths=[5], lengths_kv=[3], seed=41)
    out, mx, sm = O.prefill(case.q, case.k, case.v, case.cu_q, case.cu_kv, Nq=2, Nkv=1, D=8,
                            scale=0.3, causal=True, dtype=OR.BF16)
    out, mx, sm = out.reshape(5, 2, 8), mx.reshape(5, 2), sm.reshape(5, 2)
    assert np.all(out[:2] == 0) and np.all(mx[:2] == -np.inf) and np.all(sm[:2] == 0)
    assert np.all(sm[2:] >= 1.0)
    del rng


# ------------------------------------------------------------------ generator conventions
def pin_blocknum_worked_example(O=None):
    """aclnnMlaPrologV3WeightNz, BlockNum row: cumulative [47,151,261,422], blockSize 128 -> 5."""
    g = golden("mla_prolog_blocknum.json")
    lengths = W.lengths_from_cumulative_ends(g["cumulative_seq_lens"])
    assert lengths.tolist() == g["per_batch_lengths"]
    assert W.pool_blocks(lengths, g["block_size"]) == g["block_num"]


def pin_cumulative_seqlen_example(O=None):
    """aclnnFlashAttentionScoreV4: lengths [2,2,0,2,2] are passed as [2,4,4,6,8]."""
    g = golden("fas_v4_actual_seq_qlen.json")
    cu = W.cumulative(g["per_sequence_lengths"])
    assert cu[0] == 0 and cu[1:].tolist() == g["actual_seq_qlen"]


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
