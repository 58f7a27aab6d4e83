"""The C-ABI library loads and exports every entry point include/csa2.h declares; host-side
checks that need no GPU (no compute call is made here)."""
import ctypes as C
import re
from pathlib import Path

import pytest

import compressed_sparse_attention_03_gb300 as csa2
from compressed_sparse_attention_03_gb300 import build

HEADER = Path(__file__).resolve().parent.parent / "include" / "csa2.h"


@pytest.fixture(scope="module")
def lib():
    build.build()
    return csa2.lib()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("csa2_write_cache", "csa2_index_topk", "csa2_attend", "csa2_create", "csa2_destroy",
              "csa2_workspace_bytes", "csa2_status_string", "csa2_default_config"):
        assert n in names
    assert set(names) == set(csa2.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_status_strings_and_config_checks(lib):
    assert lib.csa2_status_string(0) == b"ok"
    assert lib.csa2_status_string(4) == b"workspace too small"
    assert lib.csa2_status_string(7) == b"batch exceeds the fixed scratch of csa2_attend_static"
    assert lib.csa2_status_string(8) == b"a bounded wait inside a kernel gave up"
    cfg = csa2.csa2_config()
    lib.csa2_default_config(C.byref(cfg))
    assert (cfg.heads, cfg.head_dim, cfg.rope_dims, cfg.idx_heads, cfg.idx_dim, cfg.window, cfg.topk, cfg.ratio) == \
        (64, 512, 64, 32, 128, 128, 512, 2)
    assert cfg.rope_base == 10000.0 and cfg.eps == 1e-20
    h = C.c_void_p()
    cfg.topk = 256   # the kernels are built for top-512 only
    assert lib.csa2_create(C.byref(cfg), C.byref(h)) == 5 and not h.value
    lib.csa2_default_config(C.byref(cfg))
    cfg.ratio = 3    # compression ratio 1 or 2 only
    assert lib.csa2_create(C.byref(cfg), C.byref(h)) == 5 and not h.value
    lib.csa2_default_config(C.byref(cfg))
    cfg.rope_base = 0.5
    assert lib.csa2_create(C.byref(cfg), C.byref(h)) == 1
    assert lib.csa2_create(None, C.byref(h)) == 1
    # no handle: every entry point refuses before touching the GPU (and launches nothing)
    launches = lib.csa2_kernel_launches()
    assert lib.csa2_workspace_bytes(None, 1, 1, 1, 10) == 0
    assert lib.csa2_index_topk(*([None] * 5), 0, None, 1, 1, None, None, None, 0, None) == 1
    assert lib.csa2_attend_static(*([None] * 5), 0, None, None, None, 1, 1, None, None) == 1
    assert lib.csa2_index_pool(*([None] * 5), 0, None, 1, 1, None, None, None, None, 0, None) == 1
    assert lib.csa2_reindex_topk(*([None] * 5), 0, None, 1, 1, None, None, None, None, 0, None) == 1
    assert lib.csa2_check(None, None) == 1
    assert lib.csa2_selftest_timeout(None, None) == 1
    assert lib.csa2_set_device_positions(None, None, 0) == 1
    assert lib.csa2_kernel_launches() == launches


class _FakeHandle:
    def __init__(self, ratio=2, dev_p0_max=None):
        self.ratio, self.dev_p0_max = ratio, dev_p0_max


def test_binding_positions_host_logic():
    """The binding's position marshalling: host arrays as int64[B] (a scalar broadcast), None
    passed as NULL only while the handle reads device positions, and workspace sizing from the
    host positions or else from the device positions' bound."""
    from compressed_sparse_attention_03_gb300 import _host_p0, _max_entries, _p0_ptr
    h = _FakeHandle()
    a = _host_p0([5, 9], 2, h)
    assert a.dtype.name == "int64" and list(a) == [5, 9]
    assert list(_host_p0(7, 3, h)) == [7, 7, 7]
    with pytest.raises(ValueError):
        _host_p0([1, 2, 3], 2, h)
    with pytest.raises(ValueError):  # host positions are required without device positions
        _host_p0(None, 2, h)
    assert _max_entries(h, a, 4) == (9 + 4) // 2
    hd = _FakeHandle(ratio=1, dev_p0_max=1000)
    assert _host_p0(None, 2, hd) is None and _p0_ptr(None) is None
    assert _max_entries(hd, None, 1) == 1001
    assert list(_host_p0([3, 4], 2, hd)) == [3, 4]  # still accepted (the library does not read it)
