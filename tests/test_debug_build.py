"""The debug build (libfattn_debug.so, compiled with -DFATTN_DEBUG): host-side checks that run
anywhere.  Its device-side rules are pinned at compile time (static_assert cases in
sm103a_ptx.cuh, so the build itself fails if a rule function is wrong); here: both libraries build,
export the same declared boundary, say which build they are, and the release build's record reads
as empty without touching a device.  The GPU side (every entry point through the debug build, no
rule broken, results equal to the release build's) is tests/test_debug_checks.py.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fattn.h")


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(fattn_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libs():
    from exact_attention_31_gb300 import _build
    _build.build_all()
    out = {}
    for name, path in (("release", _build.LIB), ("debug", _build.DEBUG_LIB)):
        L = ctypes.CDLL(path)
        L.fattn_debug_build.restype = ctypes.c_int
        L.fattn_debug_take.restype = ctypes.c_int
        L.fattn_debug_take.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(ctypes.c_ulonglong)]
        L.fattn_status_string.restype = ctypes.c_char_p
        L.fattn_status_string.argtypes = [ctypes.c_int]
        out[name] = L
    return out


def test_both_builds_export_the_declared_boundary(libs):
    names = declared_functions()
    assert "fattn_debug_build" in names and "fattn_debug_take" in names
    for which, L in libs.items():
        for name in names:
            assert hasattr(L, name), f"{which} build does not export {name}"


def test_builds_say_which_they_are(libs):
    assert libs["release"].fattn_debug_build() == 0
    assert libs["debug"].fattn_debug_build() == 1


def test_release_record_is_empty_without_a_device(libs):
    L = libs["release"]
    rules, first = ctypes.c_uint(7), ctypes.c_ulonglong(9)
    assert L.fattn_debug_take(ctypes.byref(rules), ctypes.byref(first)) == 0
    assert rules.value == 0 and first.value == 0
    # NULL arguments are rejected by both builds before anything else
    for L in libs.values():
        assert L.fattn_debug_take(None, ctypes.byref(first)) == 1
        assert L.fattn_debug_take(ctypes.byref(rules), None) == 1


def test_debug_status_has_a_name(libs):
    for L in libs.values():
        assert L.fattn_status_string(5) == b"FATTN_ERR_DEBUG"


def test_debug_build_compiles_the_checks_in():
    # the checks sit in the wrappers every kernel file uses; the debug objects are built from the
    # same sources with -DFATTN_DEBUG, and only the debug library carries the per-file records
    from exact_attention_31_gb300 import _build
    assert _build.DEBUG_FLAGS == ["-DFATTN_DEBUG"]
    assert _build.up_to_date(debug=True) and _build.up_to_date(debug=False)
    text = open(os.path.join(ROOT, "exact_attention_31_gb300", "csrc", "sm103a_ptx.cuh")).read()
    for wrapper in ("tma_load_3d", "tma_reduce_add_3d", "bulk_load", "tmem_ld_32x32b_x32", "tmem_st_32x32b_x32",
                    "mma_ss_lead", "mma_ts_lead", "mbar_arrive"):
        body = text[text.index(f"void {wrapper}(") if f"void {wrapper}(" in text else text.index(wrapper):]
        body = body[:body.index("\n}\n")]
        assert "FATTN_DBG_SKIP_IF" in body or "dbg_fails" in body, wrapper
