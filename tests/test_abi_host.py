"""Host-side checks of the C ABI that need no GPU.

The library loads, exports every entry point that ``include/nspack.h``
declares, and rejects bad arguments on the host before touching the device.
"""
import ctypes as C
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?[\w ]+?\**\s*\b(ns_\w+)\s*\(", src, flags=re.M))
    return names


@pytest.fixture(scope="module")
def nspack():
    import __graft_entry__
    __graft_entry__.build()
    import deterministic_packed_assembly_gb300 as m
    return m


def test_library_exports_every_declared_symbol(nspack):
    declared = _declared_symbols()
    assert {"ns_pack_init", "ns_pack_step", "ns_pack_fingerprint"} <= declared
    lib = C.CDLL(nspack.LIB_PATH)
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared == set(nspack.SYMBOLS)


def test_strerror(nspack):
    assert nspack.ns_pack_strerror(0) == "ok"
    for code in range(-7, 0):
        assert nspack.ns_pack_strerror(code) != "unknown error"


def _cfg(nspack, **kw):
    L = nspack._lib
    keep = dict(tok=np.zeros(64, np.int32), off=np.asarray([0, 10, 20], np.int64),
                sdb=np.asarray([0, 2], np.uint32), ssrc=np.zeros(1, np.uint32),
                sw=np.ones(1, np.uint32), tw=np.ones(1, np.uint32),
                bp=np.zeros(1, np.uint16))
    c = L.ns_pack_config()
    # host pointers stand in for device ones: every check below fails before use
    c.tokens = keep["tok"].ctypes.data & ~15
    c.n_tokens = 64
    c.doc_offsets = keep["off"].ctypes.data
    c.n_docs = 2
    c.n_sources = 1
    c.n_streams = 1
    c.T = 16
    c.stream_doc_begin = keep["sdb"].ctypes.data
    c.stream_source = keep["ssrc"].ctypes.data
    c.source_weight = keep["sw"].ctypes.data
    c.stream_weight = keep["tw"].ctypes.data
    c.source_heldout_bp = keep["bp"].ctypes.data
    c.B = 2
    c.max_steps = 4
    for k, v in kw.items():
        setattr(c, k, v)
    return c, keep


@pytest.mark.parametrize("field,value", [
    ("T", 0), ("T", 8), ("T", 24), ("T", (1 << 24) + 16), ("B", 0), ("max_steps", 0),
    ("max_steps", 1 << 30), ("n_sources", 0), ("n_streams", 0), ("n_streams", 70000),
    ("flags", 64), ("flags", 32), ("window_segment", (1 << 24) + 1), ("n_tokens", 1 << 47), ("tokens", None), ("doc_offsets", None), ("stream_doc_begin", None),
])
def test_init_rejects_bad_recipe(nspack, field, value):
    c, keep = _cfg(nspack, **{field: value})
    with pytest.raises(nspack.NsPackError) as e:
        nspack.ns_pack_init(c)
    assert e.value.code == nspack.NS_ERR_INVALID_ARG


def test_init_rejects_bad_tables(nspack):
    for name, arr in (("sw", np.zeros(1, np.uint32)), ("tw", np.zeros(1, np.uint32)),
                      ("bp", np.asarray([10001], np.uint16)),
                      ("ssrc", np.asarray([1], np.uint32)),
                      ("sdb", np.asarray([0, 3], np.uint32))):
        c, keep = _cfg(nspack)
        keep[name] = arr
        field = dict(sw="source_weight", tw="stream_weight", bp="source_heldout_bp",
                     ssrc="stream_source", sdb="stream_doc_begin")[name]
        setattr(c, field, arr.ctypes.data)
        with pytest.raises(nspack.NsPackError) as e:
            nspack.ns_pack_init(c)
        assert e.value.code == nspack.NS_ERR_INVALID_ARG, name


def test_init_rejects_misaligned_tokens(nspack):
    c, keep = _cfg(nspack)
    c.tokens = c.tokens + 4
    with pytest.raises(nspack.NsPackError) as e:
        nspack.ns_pack_init(c)
    assert e.value.code == nspack.NS_ERR_INVALID_ARG


def test_init_rejects_misaligned_offsets_and_loss_starts(nspack):
    # device offsets are read as int64 and loss starts as int32: a pointer not
    # aligned for its type is refused before anything is enqueued (without the
    # check, init would go on to the CUDA calls, which fail here otherwise)
    c, keep = _cfg(nspack)
    c.doc_offsets = c.doc_offsets + 4
    with pytest.raises(nspack.NsPackError) as e:
        nspack.ns_pack_init(c)
    assert e.value.code == nspack.NS_ERR_INVALID_ARG
    c, keep = _cfg(nspack)
    keep["ls"] = np.zeros(4, np.int32)
    c.loss_start = (keep["ls"].ctypes.data & ~3) + 2
    with pytest.raises(nspack.NsPackError) as e:
        nspack.ns_pack_init(c)
    assert e.value.code == nspack.NS_ERR_INVALID_ARG


def test_quota_noalloc_rejects_misaligned_tables(nspack):
    L = nspack._lib
    sw = np.ones(2, np.uint32)
    ss = np.asarray([0, 1], np.uint32)
    tw = np.ones(2, np.uint32)
    buf = np.zeros(64, np.int32)
    good = buf.ctypes.data & ~15
    for q, cm in ((good + 2, good + 16), (good, good + 17)):
        rc = L.lib.ns_pack_quota_noalloc(sw.ctypes.data, 2, ss.ctypes.data, tw.ctypes.data, 2,
                                         4, 3, q, cm, None)
        assert rc == nspack.NS_ERR_INVALID_ARG


def test_packer_refuses_outputs_it_would_misread_or_write_past(nspack):
    # the binding hands the library bare pointers: a tensor of the wrong type,
    # not contiguous, or smaller than the call writes is refused first
    import torch
    from deterministic_packed_assembly_gb300.packer import Packer
    T, B = 16, 4

    def out(n, r, **over):
        o = dict(tokens=torch.zeros(n, r, T, dtype=torch.int32),
                 pos=torch.zeros(n, r, T, dtype=torch.int32),
                 doc=torch.zeros(n, r, T, dtype=torch.int32),
                 mask=torch.zeros(n, r, T, dtype=torch.uint8),
                 row_fp=torch.zeros(n, r, dtype=torch.int64),
                 row_learned=torch.zeros(n, r, dtype=torch.int32))
        o.update(over)
        return o

    o = Packer.prepare(out(2, B))
    assert (o.nspack_positions, o.nspack_rows) == (2 * B * T, 2 * B)
    for bad in (dict(row_fp=torch.zeros(2, B, dtype=torch.int32)),
                dict(mask=torch.zeros(2, B, T, dtype=torch.int32)),
                dict(row_len=torch.zeros(2, B, dtype=torch.int64)),
                dict(tokens=torch.zeros(2, 2 * B, T, dtype=torch.int32)[:, ::2]),
                dict(pos=torch.zeros(2, 2 * B, T, dtype=torch.int32)[:, :B])):
        with pytest.raises(nspack.NsPackError) as e:
            Packer.prepare(out(2, B, **bad))
        assert e.value.code == nspack.NS_ERR_INVALID_ARG, list(bad)
    # the call's size against the buffers' (host checks only: no context)
    pk = Packer.__new__(Packer)
    pk.device, pk.T, pk.B, pk.schedule, pk.stream, pk._ctx = (
        torch.device("cpu"), T, B, None, None, None)
    for kw in (dict(n_steps=3, out=out(2, B)), dict(rows=(0, B), out=out(1, B - 1)),
               dict(n_steps=2, out=out(1, 2 * B, row_fp=torch.zeros(1, B, dtype=torch.int64)))):
        with pytest.raises(nspack.NsPackError) as e:
            pk.step(0, **kw)
        assert e.value.code == nspack.NS_ERR_INVALID_ARG


def test_null_context_is_rejected(nspack):
    L = nspack._lib
    out = L.ns_pack_out()
    assert L.lib.ns_pack_step(None, 0, 1, 0, 1, C.byref(out), None) == nspack.NS_ERR_INVALID_ARG
    v = C.c_uint64()
    assert L.lib.ns_pack_fingerprint(None, None, 1, C.byref(v), None) == nspack.NS_ERR_INVALID_ARG
    info = L.ns_pack_info_t()
    assert L.lib.ns_pack_info(None, C.byref(info)) == nspack.NS_ERR_INVALID_ARG
    assert L.lib.ns_pack_check(None) == nspack.NS_ERR_INVALID_ARG
    assert L.lib.ns_pack_batch_fp(None, None, 1, 1, None, None) == nspack.NS_ERR_INVALID_ARG
    assert L.lib.ns_pack_step_learned(None, None, 1, 1, None, None) == nspack.NS_ERR_INVALID_ARG
    L.lib.ns_pack_free(None)


def test_binding_structs_match_the_header_layout(nspack, tmp_path):
    # the ctypes structures of the binding and the C structures of the header
    # agree field by field: a C program built against the header prints each
    # field's offset and each structure's size
    from deterministic_packed_assembly_gb300 import _lib as L
    structs = {"ns_pack_config": L.ns_pack_config, "ns_pack_out": L.ns_pack_out,
               "ns_pack_info_t": L.ns_pack_info_t}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "nspack.h"',
             'int main(void) {']
    for name, cls in structs.items():
        lines.append(f'  printf("{name} sizeof %zu\\n", sizeof({name}));')
        for f, _ in cls._fields_:
            lines.append(f'  printf("{name} {f} %zu\\n", offsetof({name}, {f}));')
    lines += ['  return 0;', '}']
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    import subprocess
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src),
                           "-o", str(exe)])
    got = {}
    for ln in subprocess.check_output([str(exe)], text=True).splitlines():
        s, f, v = ln.split()
        got[(s, f)] = int(v)
    for name, cls in structs.items():
        assert got[(name, "sizeof")] == C.sizeof(cls), name
        for f, _ in cls._fields_:
            assert got[(name, f)] == getattr(cls, f).offset, (name, f)
