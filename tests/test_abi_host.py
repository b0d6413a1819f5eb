"""Host-only checks of the C interface: the library builds and loads, exports
every function include/fia.h declares, and rejects bad arguments with the
documented codes before touching a device."""
import ctypes
import re
import subprocess

import pytest

NULLPTR, INVALID = 161001, 161002


def test_library_exports_every_declared_function(F, built_lib):
    names = F.header_functions()
    assert {"fia_decode", "fia_prefill", "ring_attention_update", "fia_decode_workspace_size",
            "fia_prefill_workspace_size", "fia_last_error", "fia_device_status"} <= set(names)
    nm = subprocess.run(["nm", "-D", "--defined-only", built_lib], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\sT\s+(\w+)$", nm.stdout, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"


def test_library_does_not_link_the_oracle(built_lib):
    nm = subprocess.run(["nm", "-D", built_lib], capture_output=True, text=True, check=True)
    assert "oracle_" not in nm.stdout
    ldd = subprocess.run(["ldd", built_lib], capture_output=True, text=True)
    assert "liboracle" not in ldd.stdout


P = 0x10000  # a non-null, 256-byte aligned fake device address (never dereferenced)


def _decode(lib, **kw):
    a = dict(q=P, q_dtype=2, k=P, v=P, kv_dtype=2, bt=P, bt_stride=4, lens=P, max_kv_len=64, B=2, Nq=4, Nkv=2,
             D=64, bs=16, num_blocks=8, scale=0.125, aqs=None, aqo=None, sink=None, out=P, mx=None, sm=None,
             splits=0, ws=P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.fia_decode(a["q"], a["q_dtype"], a["k"], a["v"], a["kv_dtype"], a["bt"], a["bt_stride"], a["lens"],
                          a["max_kv_len"], a["B"], a["Nq"], a["Nkv"], a["D"], a["bs"], a["num_blocks"], a["scale"],
                          a["aqs"], a["aqo"], a["sink"], a["out"], a["mx"], a["sm"], a["splits"], a["ws"],
                          a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), NULLPTR), (dict(k=None), NULLPTR), (dict(bt=None), NULLPTR), (dict(lens=None), NULLPTR),
    (dict(out=None), NULLPTR), (dict(ws=None), NULLPTR), (dict(kv_dtype=3), NULLPTR),     # int8 without scale
    (dict(q_dtype=0), INVALID), (dict(q_dtype=3), INVALID), (dict(kv_dtype=1), INVALID),  # fp16 kv, bf16 q
    (dict(Nq=6, Nkv=4), INVALID), (dict(Nq=64, Nkv=2), INVALID), (dict(Nq=300, Nkv=300), INVALID),
    (dict(Nq=32, Nkv=2, kv_dtype=3, aqs=P, bs=32), INVALID),                             # int8, group 16
    (dict(D=96), INVALID), (dict(D=256), INVALID), (dict(bs=0), INVALID), (dict(bs=24), INVALID),
    (dict(bs=1024), INVALID), (dict(kv_dtype=3, aqs=P, bs=16), INVALID),                  # int8 needs bs % 32
    (dict(kv_dtype=3, aqs=P, bs=32, sink=P), INVALID),                                      # sink + int8
    (dict(bt_stride=3), INVALID), (dict(num_blocks=0), INVALID), (dict(B=70000), INVALID),
    (dict(max_kv_len=-1), INVALID), (dict(splits=-1), INVALID), (dict(scale=float("inf")), INVALID),
    (dict(q=P + 8), INVALID), (dict(k=P + 2), INVALID), (dict(ws=P + 16), INVALID),
])
def test_decode_rejects(F, kw, code):
    lib = F.library()
    assert _decode(lib, **kw) == code
    assert lib.fia_last_error()


def _noalloc(lib, **kw):
    a = dict(q=P, q_dtype=2, k=P, v=P, kv_dtype=2, bt=P, bt_stride=4, lens=P, max_kv_len=64, B=2, Nq=4, Nkv=2,
             D=64, bs=16, num_blocks=8, scale=0.125, aqs=None, aqo=None, sink=None, out=P, mx=None, sm=None,
             splits=0, stream=None)
    a.update(kw)
    return lib.fia_decode_noalloc(a["q"], a["q_dtype"], a["k"], a["v"], a["kv_dtype"], a["bt"], a["bt_stride"],
                                  a["lens"], a["max_kv_len"], a["B"], a["Nq"], a["Nkv"], a["D"], a["bs"],
                                  a["num_blocks"], a["scale"], a["aqs"], a["aqo"], a["sink"], a["out"], a["mx"],
                                  a["sm"], a["splits"], a["stream"])


@pytest.mark.parametrize("kw", [
    dict(out=None), dict(q=None), dict(lens=None), dict(kv_dtype=3), dict(out=None, D=96), dict(q=None, q_dtype=0),
    dict(q_dtype=0), dict(kv_dtype=1), dict(Nq=6, Nkv=4), dict(D=96), dict(bs=24), dict(bt_stride=3),
    dict(kv_dtype=3, aqs=P, bs=32, sink=P), dict(q=P + 8), dict(scale=float("inf")), dict(splits=-1),
])
def test_noalloc_reports_the_codes_of_fia_decode(F, kw):
    """The allocation-free entry point checks its arguments as fia_decode does, in the same
    order: the same bad argument gives the same code and message from both."""
    lib = F.library()
    rc = _decode(lib, **kw)
    msg = lib.fia_last_error()
    assert rc in (NULLPTR, INVALID)
    assert _noalloc(lib, **kw) == rc
    assert lib.fia_last_error() == msg


def test_rau_rejects(F):
    lib = F.library()
    assert lib.ring_attention_update(None, P, P, P, P, P, 2, 4, 8, 64, P, P, P, None) == NULLPTR
    assert lib.ring_attention_update(P, P, P, P, P, P, 3, 4, 8, 64, P, P, P, None) == INVALID
    assert lib.ring_attention_update(P, P, P, P, P, P, 2, 4, 8, 60, P, P, P, None) == INVALID
    assert lib.ring_attention_update(P, P, P, P, P, P, 2, 4, 300, 64, P, P, P, None) == INVALID
    assert lib.ring_attention_update(P, P, P, P, P, P, 2, 4, 8, 776, P, P, P, None) == INVALID


def test_workspace_size_needs_output(F):
    lib = F.library()
    assert lib.fia_decode_workspace_size(2, 4, 2, 64, 64, 16, 0, None) == NULLPTR
    n = ctypes.c_size_t(0)
    assert lib.fia_decode_workspace_size(2, 4, 2, 96, 64, 16, 0, ctypes.byref(n)) == INVALID


def test_options_structs_match_the_header(F, tmp_path):
    """The binding's ctypes mirrors of fia_decode_options and fia_prefill_options have the
    C layout: size and every field's offset, as gcc lays the header's structs out."""
    import os
    from attention_ifa_fia_gb300 import _binding as B
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    structs = {"fia_decode_options": B.DecodeOptions, "fia_prefill_options": B.PrefillOptions}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "fia.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'  printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", inc, str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {tuple(l.split()[:2]): int(l.split()[2]) for l in out if l}
    for cname, cls in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for fname, _ in cls._fields_:
            assert got[(cname, fname)] == getattr(cls, fname).offset, (cname, fname)


def _decode_ex(lib, B_, opts, **kw):
    a = dict(q=P, q_dtype=2, k=P, v=P, kv_dtype=2, bt=P, bt_stride=4, lens=P, max_kv_len=64, B=2, Nq=4, Nkv=2,
             D=64, bs=16, num_blocks=8, scale=0.125, aqs=None, aqo=None, sink=None, out=P, mx=None, sm=None,
             splits=0, ws=P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.fia_decode_ex(a["q"], a["q_dtype"], a["k"], a["v"], a["kv_dtype"], a["bt"], a["bt_stride"], a["lens"],
                             a["max_kv_len"], a["B"], a["Nq"], a["Nkv"], a["D"], a["bs"], a["num_blocks"], a["scale"],
                             a["aqs"], a["aqo"], a["sink"], a["out"], a["mx"], a["sm"], a["splits"], a["ws"],
                             a["ws_bytes"], a["stream"], ctypes.byref(opts))


@pytest.mark.parametrize("fields,kw,code", [
    (dict(kv_layout=2), {}, INVALID),                                  # unknown layout
    (dict(antiquant_mode=2), {}, INVALID),                             # unknown antiquant mode
    (dict(antiquant_mode=1), {}, INVALID),                             # per-tensor without int8 KV
    (dict(atten_mask=P, atten_mask_stride=63), {}, INVALID),           # mask rows shorter than max_kv_len
    (dict(quant_offset2=P), {}, INVALID),                              # offset without scale
    (dict(quant_scale2=P, quant2_per_channel=2), {}, INVALID),
    (dict(band=1, pre_tokens=3, next_tokens=-4), {}, INVALID),         # a band holding no key
    (dict(q_len=17), {}, INVALID),                                     # more query positions than built
    (dict(q_len=-1), {}, INVALID),
    (dict(q_len=9), {}, INVALID),                                      # G 2 x 9 positions > 16
    (dict(q_len=5), dict(kv_dtype=3, aqs=P, bs=32), INVALID),          # int8: G 2 x 5 > 8
    (dict(q_len=2, band=1, pre_tokens=10, next_tokens=0), {}, INVALID),  # positions with a band
    (dict(q_len=2, atten_mask=P, atten_mask_stride=64), {}, INVALID),  # positions with attenMask
])
def test_decode_ex_rejects(F, fields, kw, code):
    from attention_ifa_fia_gb300 import _binding as B
    lib = F.library()
    opts = B.DecodeOptions()
    for k, v in fields.items():
        setattr(opts, k, v)
    assert _decode_ex(lib, None, opts, **kw) == code
    assert lib.fia_last_error()


def _prefill_ex(lib, opts, **kw):
    a = dict(q=P, k=P, v=P, dtype=2, cu_q=P, cu_kv=P, B=2, T=100, Tkv=100, msq=64, mskv=64, Nq=4, Nkv=2, D=128,
             scale=0.088, mask=3, sink=None, out=P, mx=None, sm=None, ws=P, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.fia_prefill_ex(a["q"], a["k"], a["v"], a["dtype"], a["cu_q"], a["cu_kv"], a["B"], a["T"], a["Tkv"],
                              a["msq"], a["mskv"], a["Nq"], a["Nkv"], a["D"], a["scale"], a["mask"], a["sink"],
                              a["out"], a["mx"], a["sm"], a["ws"], a["ws_bytes"], a["stream"],
                              None if opts is None else ctypes.byref(opts))


@pytest.mark.parametrize("fields,kw,code", [
    (None, dict(mask=4), NULLPTR),                                                   # band without options
    (dict(pre_tokens=2, next_tokens=-3), dict(mask=4), INVALID),                     # empty band
    ({}, dict(mask=2), INVALID),                                                     # leftUpCausal: not built
    (dict(quant_offset2=P), {}, INVALID),                                            # offset without scale
    (dict(quant_scale2=P, quant2_per_channel=2), {}, INVALID),                       # per channel not 0 / 1
    (dict(block_table=P, bt_stride=1, block_size=128, num_blocks=4), dict(cu_kv=None), NULLPTR),  # no seq_lens_kv
    (dict(block_table=P, bt_stride=1, seq_lens_kv=P, block_size=24, num_blocks=4), {}, INVALID),  # not % 16
    (dict(block_table=P, bt_stride=1, seq_lens_kv=P, block_size=8, num_blocks=4), {}, INVALID),
    ({}, dict(D=96), INVALID), ({}, dict(D=256), INVALID),                           # D outside {64, 128}
    (dict(block_table=P, bt_stride=1, seq_lens_kv=P, block_size=640, num_blocks=4), {}, INVALID),
    (dict(block_table=P, bt_stride=1, seq_lens_kv=P, block_size=128, num_blocks=0), {}, INVALID),
    (dict(block_table=P, bt_stride=1, seq_lens_kv=P, block_size=128, num_blocks=4, kv_layout=5), {}, INVALID),
    (dict(block_table=P, bt_stride=1, seq_lens_kv=P, block_size=128, num_blocks=4), dict(mskv=129), INVALID),
])
def test_prefill_ex_rejects(F, fields, kw, code):
    from attention_ifa_fia_gb300 import _binding as B
    lib = F.library()
    opts = None
    if fields is not None:
        opts = B.PrefillOptions()
        for k, v in fields.items():
            setattr(opts, k, v)
    assert _prefill_ex(lib, opts, **kw) == code
    assert lib.fia_last_error()


def test_binding_checks_the_out_dtype(F):
    """The binding refuses an out tensor whose dtype is not the one the call writes: int8 with
    quant_scale2, the query's dtype without (checked before any pointer is passed on)."""
    import torch
    q = torch.zeros((3, 2, 64), dtype=torch.bfloat16)
    cu = torch.tensor([0, 3], dtype=torch.int64)
    with pytest.raises(ValueError):
        F.fia_prefill(q, q, q, cu, cu, max_seqlen_q=3, max_seqlen_kv=3, num_heads=2,
                      out=torch.empty((3, 2, 64), dtype=torch.bfloat16), quant_scale2=torch.ones(1))
    with pytest.raises(ValueError):
        F.fia_prefill(q, q, q, cu, cu, max_seqlen_q=3, max_seqlen_kv=3, num_heads=2,
                      out=torch.empty((3, 2, 64), dtype=torch.int8))
    kc = torch.zeros((2, 2, 16, 64), dtype=torch.bfloat16)
    bt = torch.zeros((3, 1), dtype=torch.int32)
    lens = torch.ones(3, dtype=torch.int64)
    with pytest.raises(ValueError):
        F.fia_decode(q, kc, kc, bt, lens, max_kv_len=16, num_heads=2,
                     out=torch.empty((3, 2, 64), dtype=torch.bfloat16), quant_scale2=torch.ones(1))
    with pytest.raises(ValueError):
        F.fia_decode(q, kc, kc, bt, lens, max_kv_len=16, num_heads=2, out=torch.empty((3, 2, 64), dtype=torch.float16))
