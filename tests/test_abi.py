"""The C-ABI library builds, loads and exports every entry point of include/dcp.h.

CPU only: host-side argument validation is exercised (it returns before
anything is launched); no kernel is run.
"""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def built():
    from context_paged_decode_gb300 import build
    return build.build_all()


def header_symbols():
    txt = open(os.path.join(ROOT, "include", "dcp.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int)\s+(dcp_\w+)\s*\(", txt, re.M)))


def test_header_lists_the_entry_points():
    syms = header_symbols()
    import context_paged_decode_gb300 as dcp
    assert syms == sorted(dcp.exported_symbols())
    assert len(syms) >= 15


def test_library_exports_every_symbol(built):
    import context_paged_decode_gb300 as dcp
    lib = C.CDLL(built[0])
    for s in header_symbols():
        assert hasattr(lib, s), s
    dcp.load()
    assert dcp.load().dcp_version() == 100
    assert dcp.load().dcp_strerror(-1) == b"invalid argument or layout"
    assert dcp.load().dcp_strerror(-2).startswith(b"workspace")


def test_missing_library_fails_loudly(tmp_path):
    import context_paged_decode_gb300 as dcp
    saved = dcp._lib
    dcp._lib = None
    try:
        with pytest.raises(dcp.DcpError):
            dcp.load(str(tmp_path / "nope.so"))
    finally:
        dcp._lib = saved


def test_host_validation_rejects_bad_layouts(built):
    import context_paged_decode_gb300 as dcp
    lib = dcp.load()
    bad = [dcp.Layout(0, 16, 1), dcp.Layout(17, 16, 1), dcp.Layout(2, 16, 3),
           dcp.Layout(2, 0, 1), dcp.Layout(2, 16, 0)]
    for L in bad:
        assert lib.dcp_local_seq_lens(L, None, 1, None, None, None) == -1
        assert lib.dcp_slot_mapping(L, None, None, 1, None, 1, 1, 0, 1, None, None, None,
                                    None) == -1
        n = C.c_size_t(0)
        assert lib.dcp_decode_workspace_size(L, 0, 1, 8, 2, 64, C.byref(n)) == -1
    L = dcp.Layout(2, 16, 1)
    # empty work is a no-op success; null pointers with work are rejected
    assert lib.dcp_local_seq_lens(L, None, 0, None, None, None) == 0
    assert lib.dcp_local_seq_lens(L, None, 3, None, None, None) == -1
    # GQA: Hq not a multiple of Hkv, unsupported head_dim
    kv = dcp.PagedKVStruct()
    assert lib.dcp_decode_gqa(L, C.c_void_p(16), 1, 6, 4, 128, 1.0, 1, kv, C.c_void_p(16), None,
                              C.c_void_p(16), 1, None, None, 0, None, None) == -1
    assert lib.dcp_decode_gqa(L, C.c_void_p(16), 1, 8, 2, 100, 1.0, 1, kv, C.c_void_p(16), None,
                              C.c_void_p(16), 1, None, None, 0, None, None) == -1
    # merge: bad head dim
    assert lib.dcp_lse_merge(2, None, None, 1, 1, 6, None, None, 0, None, None) == -1
    # workspace sizing is a host computation
    n = C.c_size_t(0)
    assert lib.dcp_decode_workspace_size(L, 0, 4, 8, 2, 64, C.byref(n)) == 0 and n.value > 0
