"""GPU parity of ring_attention_update against the oracle's merge rule."""
import numpy as np
import pytest
import torch

import fia_workloads as W
import oracle
from parity import OUT_TOL, SUM_TOL, assert_close, assert_close_max, to_f64

pytestmark = pytest.mark.gpu

_DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def _partials(rng, rows, N, D, dtype, dev, inf_frac=0.1):
    o = torch.from_numpy(rng.standard_normal((rows, N, D), dtype=np.float32)).to(dev).to(_DT[dtype])
    m = rng.standard_normal((rows, N)).astype(np.float32) * 3
    s = rng.uniform(1.0, 50.0, (rows, N)).astype(np.float32)
    empty = rng.random((rows, N)) < inf_frac
    m[empty] = -np.inf
    s[empty] = 0.0
    o[torch.from_numpy(empty).to(dev)] = 0
    return o, torch.from_numpy(m).to(dev), torch.from_numpy(s).to(dev)


@pytest.mark.parametrize("dtype,N,D", [("bf16", 8, 128), ("fp16", 4, 64), ("fp32", 2, 768), ("bf16", 3, 8)])
def test_rau_matches_oracle(F, cuda, dtype, N, D):
    rng = np.random.default_rng(N * 1000 + D)
    rows = 257
    prev = _partials(rng, rows, N, D, dtype, cuda)
    cur = _partials(rng, rows, N, D, dtype, cuda)
    out, mx, sm = F.ring_attention_update(*prev, *cur)
    ref = oracle.rau(*(to_f64(t) for t in prev), *(to_f64(t) for t in cur))
    key = dtype if dtype != "fp32" else "fp32"
    assert_close("out", to_f64(out), ref[0], *OUT_TOL[key if key in OUT_TOL else "fp32"])
    assert_close_max("max", to_f64(mx), ref[1])
    assert_close("sum", to_f64(sm), ref[2], *SUM_TOL)


def test_rau_in_place_equals_out_of_place(F, cuda):
    rng = np.random.default_rng(5)
    prev = _partials(rng, 100, 8, 64, "bf16", cuda)
    cur = _partials(rng, 100, 8, 64, "bf16", cuda)
    a = F.ring_attention_update(*prev, *cur)
    p2 = [t.clone() for t in prev]
    F.ring_attention_update(*p2, *cur, out=p2[0], max_out=p2[1], sum_out=p2[2])
    assert torch.equal(a[0].view(torch.int16), p2[0].view(torch.int16))
    assert torch.equal(a[1], p2[1]) and torch.equal(a[2], p2[2])


def test_rau_fold_of_decode_chunks_equals_unsplit(F, cuda):
    """Four decode calls over consecutive key ranges, folded by the RAU kernel, match the oracle."""
    from parity import DeviceDecode, compare_decode, run_decode
    case = W.make_decode_case(B=3, Nq=8, Nkv=2, D=128, block_size=64, lengths=[1024, 1024, 1024], seed=23,
                              sink=True)
    dd = DeviceDecode(case)
    cols = 4
    lens = torch.full((case.B,), cols * case.block_size, dtype=torch.int64, device=cuda)
    acc = None
    for j in range(4):
        bt = dd.bt[:, j * cols:(j + 1) * cols].contiguous()
        part = run_decode(F, dd, sink=dd.sink if j == 2 else None, max_kv_len=cols * case.block_size, lens=lens,
                          bt=bt)
        acc = part if acc is None else F.ring_attention_update(*acc, *part)
    compare_decode(case, *acc)
