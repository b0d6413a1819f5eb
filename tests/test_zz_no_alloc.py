"""fia_decode_noalloc, the decode entry point for callers that cannot allocate
device memory (it keeps its workspace in a fixed array inside the library), must
give the same results as fia_decode with a caller-provided workspace.

The file name sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import fia_workloads as W
from parity import OUT_TOL, SUM_TOL, DeviceDecode, assert_close, assert_close_max, run_decode, to_f64

pytestmark = pytest.mark.gpu


def _noalloc(F, dd):
    c = dd.case
    mx = torch.full((c.B, c.Nq), float("nan"), dtype=torch.float32, device=dd.q.device)
    sm = torch.full_like(mx, float("nan"))
    out = torch.empty((c.B, c.Nq, c.D), dtype=dd.q.dtype, device=dd.q.device)
    return F.fia_decode_noalloc(dd.q, dd.k, dd.v, dd.bt, dd.lens, max_kv_len=c.max_len, num_heads=c.Nq,
                                num_kv_heads=c.Nkv, scale=c.scale, antiquant_scale=dd.aq_scale,
                                antiquant_offset=dd.aq_offset, sink=dd.sink, out=out, softmax_max=mx,
                                softmax_sum=sm)


@pytest.mark.parametrize("make", [
    lambda: W.bf16_gqa_decode(),
    lambda: W.make_decode_case(B=3, Nq=8, Nkv=2, D=64, block_size=16, dtype=W.FP16, lengths=[1, 300, 77],
                               sink=True, seed=71),
    lambda: W.make_decode_case(B=2, Nq=8, Nkv=2, D=128, block_size=64, kv_dtype=W.INT8, lengths=[900, 33],
                               seed=72),
], ids=["bf16_gqa_decode", "fp16_sink_bs16", "int8"])
def test_noalloc_matches_fia_decode_twice(F, cuda, make):
    case = make()
    dd = DeviceDecode(case)
    ref = run_decode(F, dd)  # fia_decode with a workspace allocated by the caller
    tol = OUT_TOL[case.dtype]
    for _ in range(2):      # the scratch keeps the previous call's contents; results must not depend on it
        got = _noalloc(F, dd)
        torch.cuda.synchronize()
        assert_close("out", to_f64(got[0]), to_f64(ref[0]), *tol)
        assert_close_max("softmax_max", to_f64(got[1]), to_f64(ref[1]))
        assert_close("softmax_sum", to_f64(got[2]), to_f64(ref[2]), *SUM_TOL)
    assert F.fia_device_status() == 0


def test_noalloc_rejects_problems_beyond_its_scratch(F, cuda):
    """A workspace need above the fixed scratch is refused with 161002 and a clear message."""
    case = W.make_decode_case(B=2, Nq=32, Nkv=2, D=128, block_size=16, lengths=[5, 9], seed=73)
    dd = DeviceDecode(case)
    big = 4_000_000  # KV length bound: 977 chunks x 2 x 2 items of 16 x 128 fp32 partials = 32 MB
    need = F.fia_decode_workspace_size(case.B, case.Nq, case.Nkv, case.D, big, case.block_size, 1000)
    assert need > 16 << 20
    bt = torch.zeros((case.B, big // case.block_size + 1), dtype=torch.int32, device=cuda)
    with pytest.raises(F.FiaError) as ei:
        F.fia_decode_noalloc(dd.q, dd.k, dd.v, bt, dd.lens, max_kv_len=big, num_heads=case.Nq,
                             num_kv_heads=case.Nkv, num_splits=1000)
    assert ei.value.code == 161002 and "scratch" in str(ei.value)
