"""The C-ABI library builds, loads and exports every function include/kvq.h
declares (CPU only: no compute call is made without a GPU)."""
import ctypes
import os
import re

import pytest

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


# ---- host-side validation (returns before any CUDA call: runs without a GPU) ----
OK, INVALID, UNSUPPORTED = 0, 1, 2
P = 0x100000          # a 16-byte-aligned stand-in address: validation never dereferences it


def _decode_args(**kw):
    a = dict(q=P, dtype=1, B=4, Hq=8, Hkv=2, D=128, kc=P, vc=P, ks=P, vs=P, nb=64, bs=16,
             bt=P, mb=8, cl=P, mc=128, scale=0.088, out=P, ws=None, wsb=0, stream=None)
    a.update(kw)
    return [a[k] for k in ("q", "dtype", "B", "Hq", "Hkv", "D", "kc", "vc", "ks", "vs", "nb",
                           "bs", "bt", "mb", "cl", "mc", "scale", "out", "ws", "wsb", "stream")]


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), OK),                       # nothing to do
    (dict(dtype=7), INVALID),
    (dict(Hq=0), INVALID),
    (dict(Hq=6, Hkv=4), INVALID),          # heads not a multiple of KV heads
    (dict(Hq=32, Hkv=2), UNSUPPORTED),     # group of 16
    (dict(bs=32), UNSUPPORTED),
    (dict(D=96), UNSUPPORTED),
    (dict(B=4097), UNSUPPORTED),
    (dict(scale=float("nan")), INVALID),
    (dict(q=None), INVALID),
    (dict(ks=None), INVALID),              # the INT8 decode needs scale planes
    (dict(q=P + 8), INVALID),              # q not 16-byte aligned
    (dict(mc=129), INVALID),               # bound above the block table's reach
    (dict(mb=0), INVALID),
])
def test_decode_host_validation(kw, status):
    assert kvq.load().kvq_paged_decode(*_decode_args(**kw)) == status


@pytest.mark.parametrize("kw", [dict(B=-1), dict(Hq=0), dict(Hkv=0), dict(Hq=-8),
                                dict(mc=-1)])
def test_noalloc_rejects_before_any_device_work(kw):
    """kvq_paged_decode_noalloc answers these without looking the scratch up
    (so without a device)."""
    args = _decode_args(**kw)
    del args[18:20]                        # no workspace arguments
    assert kvq.load().kvq_paged_decode_noalloc(*args) == INVALID


@pytest.mark.parametrize("kw,status", [
    (dict(T=0), OK),
    (dict(bs=8), UNSUPPORTED),
    (dict(D=80), UNSUPPORTED),
    (dict(kstride=100), INVALID),          # below num_kv_heads * head_dim
    (dict(k=None), INVALID),
    (dict(slots=P + 4), INVALID),          # int64 slots not 8-byte aligned
    (dict(dtype=3), INVALID),
])
def test_append_host_validation(kw, status):
    a = dict(k=P, v=P, kstride=256, vstride=256, T=5, Hkv=2, D=128, dtype=0, slots=P, kc=P,
             vc=P, ks=P, vs=P, nb=64, bs=16, stream=None)
    a.update(kw)
    args = [a[k] for k in ("k", "v", "kstride", "vstride", "T", "Hkv", "D", "dtype", "slots",
                           "kc", "vc", "ks", "vs", "nb", "bs", "stream")]
    assert kvq.load().kvq_quantize_append(*args) == status


@pytest.mark.parametrize("kw,status", [
    (dict(mq=0), OK),                      # no queries
    (dict(tq=0, q=None, out=None), OK),    # no query rows: q and out may be null
    (dict(tq=0, q=None, qs=None), INVALID),
    (dict(tq=-1), INVALID),
    (dict(q=None), INVALID),               # rows without q
    (dict(mq=-1), INVALID),
    (dict(qs=None), INVALID),
    (dict(D=80), UNSUPPORTED),
])
def test_prefill_host_validation(kw, status):
    a = dict(q=P, dtype=1, B=2, Hq=8, Hkv=2, D=128, kc=P, vc=P, ks=P, vs=P, nb=64, bs=16, bt=P,
             mb=8, cl=P, mc=128, qs=P, tq=64, mq=32, scale=0.088, out=P, stream=None)
    a.update(kw)
    args = [a[k] for k in ("q", "dtype", "B", "Hq", "Hkv", "D", "kc", "vc", "ks", "vs", "nb",
                           "bs", "bt", "mb", "cl", "mc", "qs", "tq", "mq", "scale", "out",
                           "stream")]
    assert kvq.load().kvq_paged_prefill(*args) == status


@pytest.mark.parametrize("kw,status", [
    (dict(B=0), OK),
    (dict(keep=-1), INVALID),
    (dict(bs=32), UNSUPPORTED),
    (dict(D=48), UNSUPPORTED),
    (dict(trim=None), INVALID),
])
def test_trim_host_validation(kw, status):
    a = dict(kc=P, vc=P, ks=P, vs=P, nb=64, bs=16, Hkv=2, D=128, bt=P, B=2, mb=8, cl=P, trim=P,
             keep=4, stream=None)
    a.update(kw)
    args = [a[k] for k in ("kc", "vc", "ks", "vs", "nb", "bs", "Hkv", "D", "bt", "B", "mb", "cl",
                           "trim", "keep", "stream")]
    assert kvq.load().kvq_trim_front_keep_sink(*args) == status


def test_workspace_size_of_invalid_shapes_is_zero():
    L = kvq.load()
    assert L.kvq_decode_workspace_bytes(0, 8, 2, 128, 1024) == 0
    assert L.kvq_decode_workspace_bytes(4, 8, 3, 128, 1024) == 0     # 8 % 3
    assert L.kvq_decode_workspace_bytes(4, 8, 2, 96, 1024) == 0      # head_dim
    assert L.kvq_decode_partition_pages(4, 64, 2, 128, 1024) == 0    # group of 32
