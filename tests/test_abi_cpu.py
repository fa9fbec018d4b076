"""The C ABI without a GPU: the library loads, exports every declared symbol,
and rejects bad arguments on the host before touching CUDA."""

import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    # Rebuild so that the library matches the sources under test.
    from sliding_window_attention_02_gb300 import _build
    _build.build()
    import sliding_window_attention_02_gb300 as rswa
    return rswa.load()


def test_every_declared_symbol_is_exported(lib):
    import sliding_window_attention_02_gb300 as rswa
    names = rswa.declared_symbols()
    assert len(names) >= 15, names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/rswa.h but not exported"
    # and the binding wraps each of them under the same name
    for name in names:
        assert hasattr(rswa, name), f"binding lacks {name}"


def test_strerror(lib):
    for code in range(0, 7):
        assert lib.rswa_strerror(code)
    assert b"unknown" in lib.rswa_strerror(99)


def test_footprint_validation(lib):
    out = ctypes.c_size_t(0)
    f = lib.rswa_cache_footprint
    assert f(16, 8, 1, 64, 1, 0, ctypes.byref(out)) == 0
    small = out.value
    # at least the K and V slabs: 2 * B*H*(m+n)*d * elt
    assert small >= 2 * 1 * 1 * 24 * 64 * 4
    assert f(288, 128, 10, 128, 1, 1, ctypes.byref(out)) == 0
    assert out.value >= 2 * 10 * 416 * 128 * 2
    assert f(16, 8, 1, 96, 1, 0, ctypes.byref(out)) == 3     # head_dim
    assert f(16, 8, 1, 64, 1, 7, ctypes.byref(out)) == 3     # dtype
    assert f(-1, 8, 1, 64, 1, 0, ctypes.byref(out)) == 1
    assert f(16, 0, 1, 64, 1, 0, ctypes.byref(out)) == 1
    assert f(16, 8, 0, 64, 1, 0, ctypes.byref(out)) == 1
    assert f(16, 8, 1, 64, 0, 0, ctypes.byref(out)) == 1
    assert f(16, 8, 1, 64, 1, 0, None) == 1


def test_create_validation_before_cuda(lib):
    out = ctypes.c_size_t(0)
    assert lib.rswa_cache_footprint(16, 8, 1, 64, 1, 0, ctypes.byref(out)) == 0
    need = out.value
    h = ctypes.c_void_p()
    create = lib.rswa_cache_create
    assert create(16, 8, 1, 64, 1, 0, None, need, ctypes.byref(h)) == 1
    assert create(16, 8, 1, 64, 1, 0, 0x1008, need, ctypes.byref(h)) == 1  # misaligned
    assert create(16, 8, 1, 64, 1, 0, 0x1000, need - 1, ctypes.byref(h)) == 2
    assert create(16, 8, 1, 96, 1, 0, 0x1000, need, ctypes.byref(h)) == 3
    assert create(16, 8, 1, 64, 1, 0, 0x1000, need, None) == 1
    # injected CUDA failure: reported before any CUDA call
    lib.rswa_debug_fail_next_cuda(1)
    assert create(16, 8, 1, 64, 1, 0, 0x1000, need, ctypes.byref(h)) == 5
    assert h.value is None


def test_bad_handles(lib):
    bogus = ctypes.c_void_p(0x1234)
    assert lib.rswa_cache_destroy(None) == 4
    assert lib.rswa_cache_destroy(bogus) == 4
    arr = (ctypes.c_int64 * 1)(4)
    assert lib.rswa_prefill(bogus, None, 16, 16, None, arr, 0, None) == 4
    assert lib.rswa_append_kv(bogus, 16, 16, None) == 4
    assert lib.rswa_decode_step(bogus, 16, 16, None, None) == 4
    assert lib.rswa_decode_step_fused(bogus, 16, 16, 16, 16, None, None) == 4
    out = ctypes.c_size_t(0)
    assert lib.rswa_cache_bytes(bogus, 0, ctypes.byref(out)) == 4
    assert lib.rswa_sync_status(bogus) == 4
    ko, vo = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.rswa_cache_kv_offsets(bogus, ctypes.byref(ko), ctypes.byref(vo)) == 4


def test_library_links_no_torch():
    # The shared library depends on no torch / python symbols.
    import sliding_window_attention_02_gb300 as rswa
    r = subprocess.run(["ldd", rswa.library_path()], capture_output=True,
                       text=True)
    assert "torch" not in r.stdout and "python" not in r.stdout


def test_build_entry_compiles(tmp_path):
    # build() is the driver's build check; it must succeed without a GPU.
    r = subprocess.run([sys.executable, "-c",
                        "import __graft_entry__ as g; g.build()"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
