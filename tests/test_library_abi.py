"""The C-ABI library builds, loads and exports every function include/kvq.h
declares (CPU only: no compute call is made without a GPU)."""
import ctypes
import os
import re

import int8_quantized_paged_tokenwise_gb300 as kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(kvq_[a-z0-9_]+)\s*\(", src))


def test_header_declarations_match_binding_list():
    assert _declared() == set(kvq.HEADER_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = kvq.load()
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_host_only_entry_points():
    assert kvq.kvq_status_string(0) == "ok"
    assert kvq.kvq_status_string(4) == "workspace too small"
    assert kvq.load().kvq_version() == 100


def test_library_is_in_tree():
    assert os.path.dirname(str(kvq.LIB_PATH)).startswith(ROOT)
