"""The C-ABI library builds, loads and exports every entry point that
include/*.h declares; host-side argument validation rejects bad calls
before any CUDA work (no GPU needed: none of these calls reaches a kernel)."""
import ctypes
import glob
import os
import re

import pytest

from conftest import ROOT

HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


@pytest.fixture(scope="module")
def lib():
    from stream_compaction_device_gb300 import build as b
    b.build()
    from stream_compaction_device_gb300 import _lib
    return _lib.load()


def declared_functions():
    names = set()
    for header in HEADERS:
        text = open(header, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:devscan_status|const char \*)\s*(\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    assert [os.path.basename(h) for h in HEADERS] == ["devscan.h", "devscan_measure.h"]
    names = declared_functions()
    assert "devscan_measure_set_carry_mode" in names
    for want in ("scan_inclusive_i32", "scan_exclusive_f32", "compact_i32", "split_bit_u32",
                 "radix_sort_u32", "devscan_device_status", "devscan_status_string"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 14
    for name in names:
        assert hasattr(lib, name), name


def test_library_is_in_tree(lib):
    from stream_compaction_device_gb300 import _lib
    assert os.path.dirname(_lib.LIB_PATH) == os.path.join(ROOT, "stream_compaction_device_gb300")


def test_status_strings(lib):
    for code in range(6):
        s = lib.devscan_status_string(code)
        assert isinstance(s, bytes) and s
    assert lib.devscan_status_string(99) == b"unknown status"


def test_validation_without_device_work(lib):
    from stream_compaction_device_gb300._lib import ERR_INVALID, ERR_UNSUPPORTED, OK
    fake = ctypes.c_void_p(4096)  # never dereferenced: every call below fails validation first
    for name in ("scan_inclusive_i32", "scan_exclusive_u32", "scan_inclusive_f32"):
        fn = getattr(lib, name)
        assert fn(None, fake, 10, 0, None) == ERR_INVALID          # null input
        assert fn(fake, None, 10, 0, None) == ERR_INVALID          # null output
        assert fn(fake, fake, 10, 7, None) == ERR_INVALID          # unknown operator
        assert fn(None, None, 0, 0, None) == OK                     # n == 0 is a no-op
    assert lib.scan_inclusive_f32(fake, fake, 10, 2, None) == ERR_UNSUPPORTED   # xor on fp32
    assert lib.scan_exclusive_i32(ctypes.c_void_p(4098), fake, 10, 0, None) == ERR_INVALID  # misaligned
    assert lib.compact_i32(fake, fake, fake, None, 10, None) == ERR_INVALID     # null count
    assert lib.compact_i32(fake, fake, fake, fake, 2**31, None) == ERR_INVALID  # n > INT32_MAX
    assert lib.compact_i32(ctypes.c_void_p(8192), ctypes.c_void_p(1 << 20), ctypes.c_void_p(8192 + 16),
                           ctypes.c_void_p(1 << 22), 100, None) == ERR_INVALID  # out overlaps in
    assert lib.split_bit_u32(fake, ctypes.c_void_p(1 << 20), 32, 10, None) == ERR_INVALID
    assert lib.split_bit_u32(fake, ctypes.c_void_p(1 << 20), -1, 10, None) == ERR_INVALID
    assert lib.split_bit_u32(fake, fake, 3, 10, None) == ERR_INVALID            # in place
    assert lib.split_bit_u32(None, None, 3, 0, None) == OK
    assert lib.radix_sort_u32(fake, fake, 10, None) == ERR_INVALID
    assert lib.radix_sort_u32(None, None, 0, None) == OK
    for name in ("scan_inclusive_host_i32", "scan_exclusive_host_f32"):
        fn = getattr(lib, name)
        assert fn(None, fake, 10, 0, fake, ctypes.c_void_p(1 << 20), None) == ERR_INVALID   # null host input
        assert fn(fake, fake, 10, 0, fake, ctypes.c_void_p(4096 + 8), None) == ERR_INVALID  # device buffers overlap
        assert fn(None, None, 0, 0, None, None, None) == OK                                # n == 0
    assert lib.scan_inclusive_host_f32(fake, fake, 10, 2, fake, fake, None) == ERR_UNSUPPORTED
    assert lib.devscan_measure_set_carry_mode(9) == ERR_INVALID
    assert lib.devscan_measure_set_carry_mode(0) == OK
    assert lib.devscan_selftest_stalled_wait(0, None) == ERR_INVALID


def test_product_path_has_no_oracle_dependency():
    """The CUDA path never imports, links or loads the oracle."""
    pkg = os.path.join(ROOT, "stream_compaction_device_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text, f
