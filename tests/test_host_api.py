"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host before any launch (no GPU needed: these calls return
before touching the device, and no device pointer is ever dereferenced)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qasa.h")


@pytest.fixture(scope="module")
def lib():
    from query_aware_sparse_append_gb300 import build
    build.build()
    from query_aware_sparse_append_gb300 import binding
    return binding


def declared_entry_points():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:qasa_status|size_t|const char \*|int32_t)\s*\*?\s*(qasa_\w+)\s*\(",
                                 text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert len(names) >= 8, names
    so = ctypes.CDLL(lib.library_path())
    for n in names:
        assert hasattr(so, n), n
    assert set(lib.EXPORTED) <= set(names)


def test_status_strings_and_version(lib):
    assert lib.version() == 100
    for code in range(0, 9):
        assert lib.status_string(code) != "unknown status"
    assert lib.status_string(99) == "unknown status"


def _cache(lib, **kw):
    f = dict(k_pool=0x10000, v_pool=0x20000, page_bounds=0x30000, num_phys_pages=64,
             num_kv_heads=4, page_size=16, head_dim=128, dtype=1)
    f.update(kw)
    return lib._Cache(f["k_pool"], f["v_pool"], f["page_bounds"], f["num_phys_pages"],
                      f["num_kv_heads"], f["page_size"], f["head_dim"], f["dtype"])


def _decode(lib, cache, **kw):
    a = dict(q=0x40000, Hq=32, bt=0x50000, maxp=512, lens=0x60000, bud=0x70000, maxb=64,
             out=0x80000, sel=0x90000, ws=0xA0000, wsb=1 << 30, batch=8)
    a.update(kw)
    return lib._lib.qasa_sparse_decode_attention(
        ctypes.byref(cache) if cache is not None else None, a["q"], a["Hq"], a["bt"], a["maxp"],
        a["lens"], a["bud"], a["maxb"], 0.0, a["out"], a["sel"], None, a["ws"], a["wsb"],
        a["batch"], None, None)


@pytest.mark.parametrize("field,value,code", [
    ("dtype", 7, 2), ("head_dim", 96, 3), ("page_size", 8, 3), ("num_kv_heads", 0, 3),
    ("k_pool", 0, 1), ("page_bounds", 0, 1), ("v_pool", 0x20008, 4),
])
def test_cache_checks(lib, field, value, code):
    assert _decode(lib, _cache(lib, **{field: value})) == code


@pytest.mark.parametrize("arg,value,code", [
    ("q", 0, 1), ("bt", 0, 1), ("lens", 0, 1), ("out", 0, 1), ("bud", 0, 1), ("sel", 0, 1),
    ("Hq", 30, 3), ("Hq", 4 * 9, 3), ("maxp", 0, 3), ("maxp", 20000, 3), ("maxb", 1, 5),
    ("q", 0x40004, 4), ("out", 0x80008, 4), ("batch", -1, 3), ("ws", 0, 6),
])
def test_decode_argument_checks(lib, arg, value, code):
    got = _decode(lib, _cache(lib), **{arg: value})
    if arg == "ws":
        # the workspace check needs the device's SM count: without a GPU the
        # library reports the failed device query instead
        assert got in (6, 7)
    else:
        assert got == code


def test_empty_batch_is_ok_without_pointers(lib):
    assert _decode(lib, _cache(lib), batch=0, q=0, out=0, sel=0, bt=0, lens=0) == 0
    assert _decode(lib, None, batch=0) == 1


def test_append_argument_checks(lib):
    c = _cache(lib)
    f = lib._lib.qasa_kv_append
    assert f(None, 1, 8, 1, None, 16, 16, 1, 1, None, None) == 1
    assert f(ctypes.byref(c), 0, 8, 0x100, None, 0x200, 0x300, 1, 1, None, None) == 1
    assert f(ctypes.byref(c), 0x100, 0, 0x100, None, 0x200, 0x300, 1, 1, None, None) == 3
    assert f(ctypes.byref(c), 0x100, 8, 0x100, None, 0x208, 0x300, 1, 1, None, None) == 4
    assert f(ctypes.byref(c), 0x100, 8, 0x100, None, 0x200, 0x300, 0, 1, None, None) == 0


def test_workspace_size_rejects_bad_shapes(lib):
    c = _cache(lib)
    assert lib._lib.qasa_decode_workspace_size(-1, 32, ctypes.byref(c), 512) == 0
    assert lib._lib.qasa_decode_workspace_size(8, 2, ctypes.byref(c), 512) == 0
    assert lib._lib.qasa_decode_workspace_size(8, 32, None, 512) == 0


def test_host_call_form_query(lib, monkeypatch):
    # direct form only when all six buffers are page-locked memory the device
    # addresses at the same pointer: a missing buffer, ordinary (pageable)
    # host memory, or QASA_HOST_DIRECT=0 give the staged form (0)
    f = lib._lib.qasa_host_call_is_direct
    bufs = [ctypes.create_string_buffer(64) for _ in range(6)]
    ptrs = [ctypes.addressof(b) for b in bufs]
    for i in range(6):
        assert f(*[None if j == i else p for j, p in enumerate(ptrs)]) == 0
    assert f(*ptrs) == 0
    monkeypatch.setenv("QASA_HOST_DIRECT", "0")
    assert f(*ptrs) == 0


def test_debug_trace_argument_checks(lib):
    n = lib.debug_trace_bytes()
    assert n == lib.TRACE_MAX_CTAS * (lib.TRACE_SELECT_EVENTS + lib.TRACE_ATTN_EVENTS) * 8
    assert lib._lib.qasa_debug_trace(0x1004, n) == 4           # QASA_ERR_ALIGN
    assert lib._lib.qasa_debug_trace(0x1000, n - 8) == 6       # QASA_ERR_WORKSPACE
    assert lib._lib.qasa_debug_trace(None, 0) == 0             # off
