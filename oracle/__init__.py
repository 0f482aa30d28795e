"""FP64 CPU oracle for tokenwise symmetric INT8 paged KV caching and decode.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library: the arithmetic lives in ``kvq_oracle.c`` (plain C,
double precision) and this module only marshals numpy arrays into it.

What it computes follows two pages:

* "feat: opt-in INT8 KV-cache quantization" (MoE-Infinity PR #183),
  sections "What landed" and "Precision & memory" -- one upward-rounded FP16
  scale per (layer, page, KV head, token), symmetric codes without -128, exact
  zero, element error at most half the stored scale plus 1e-6, INT8 payload
  plus FP16 scale plane, dequantized softmax attention as the reference.
* "fix(cuda/kv): correct Int8 KV per-token scale ..." (mlxcel PR #717),
  section "The Int8 bug and fix" -- scale is absmax/127 and becomes 1.0 only
  for an all-zero token, so the largest coordinate maps to +-127.

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts
the pages or the mathematics fix (no function is "parity unpinned").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "kvq_oracle.c"
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "libkvq_oracle.so"

_lib = None


def build(force: bool = False) -> Path:
    """Compile the C oracle with gcc (no fast-math, no FP contraction)."""
    if not force and _LIB_PATH.exists() and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime:
        return _LIB_PATH
    _BUILD.mkdir(exist_ok=True)
    tmp = _BUILD / f"libkvq_oracle.{os.getpid()}.so"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", str(tmp), str(_SRC), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(str(_LIB_PATH))
        u16, i64, i32, f64, vp = (ctypes.c_uint16, ctypes.c_int64, ctypes.c_int,
                                  ctypes.c_double, ctypes.c_void_p)
        L.orc_fp16_to_double.argtypes = [u16]; L.orc_fp16_to_double.restype = f64
        L.orc_bf16_to_double.argtypes = [u16]; L.orc_bf16_to_double.restype = f64
        L.orc_fp16_round_up.argtypes = [f64]; L.orc_fp16_round_up.restype = u16
        L.orc_fp16_from_double_rne.argtypes = [f64]; L.orc_fp16_from_double_rne.restype = u16
        L.orc_bf16_from_double_rne.argtypes = [f64]; L.orc_bf16_from_double_rne.restype = u16
        L.orc_token_scale.argtypes = [vp, i32, i32]; L.orc_token_scale.restype = u16
        L.orc_quantize_row.argtypes = [vp, i32, i32, u16, vp]; L.orc_quantize_row.restype = None
        L.orc_dequant.argtypes = [ctypes.c_int8, u16]; L.orc_dequant.restype = f64
        L.orc_quantize_rows.argtypes = [vp, i64, i32, i32, vp, vp]; L.orc_quantize_rows.restype = None
        L.orc_quantize_rows_static.argtypes = [vp, i64, i32, i32, ctypes.c_float, vp]
        L.orc_quantize_rows_static.restype = None
        L.orc_prefill_sequence.argtypes = [vp, vp, vp, i64, i64, i32, i32, i32, i32, i32, f64,
                                           vp, vp, vp, vp]
        L.orc_prefill_sequence.restype = None
        L.orc_trim_keep_sink.argtypes = [vp, i64, i64, i64, i64, vp]
        L.orc_trim_keep_sink.restype = i64
        L.orc_dequantize_rows.argtypes = [vp, vp, i64, i32, i32, vp]
        L.orc_dequantize_rows.restype = None
        L.orc_quantize_append.argtypes = [vp, vp, i64, i64, i64, i32, i32, i32, vp,
                                          vp, vp, vp, vp, i64, i32]
        L.orc_quantize_append.restype = i64
        L.orc_attend_one.argtypes = [vp, vp, vp, i64, i64, i32, f64, vp]
        L.orc_attend_one.restype = None
        L.orc_attend_one_partitioned.argtypes = [vp, vp, vp, i64, i64, i32, f64, i64, vp, vp]
        L.orc_attend_one_partitioned.restype = None
        L.orc_decode_sequence.argtypes = [vp, vp, vp, i64, i32, i32, i32, i32, i32, f64,
                                          vp, i32, vp, vp, vp, vp]
        L.orc_decode_sequence.restype = None
        L.orc_page_bytes_int8.argtypes = [i32, i32, i32]; L.orc_page_bytes_int8.restype = i64
        L.orc_page_bytes_native16.argtypes = [i32, i32, i32]
        L.orc_page_bytes_native16.restype = i64
        _lib = L
    return _lib


def _is_bf16(dtype: str) -> int:
    if dtype not in ("fp16", "bf16"):
        raise ValueError(f"dtype must be 'fp16' or 'bf16', got {dtype!r}")
    return int(dtype == "bf16")


# ---------------------------------------------------------------- scalars ---
def fp16_to_double(bits: int) -> float:
    return lib().orc_fp16_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return lib().orc_bf16_to_double(int(bits))


def bits_to_double(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact decode of a 16-bit pattern array to float64."""
    f = lib().orc_bf16_to_double if _is_bf16(dtype) else lib().orc_fp16_to_double
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    return np.array([f(int(b)) for b in flat], dtype=np.float64).reshape(np.shape(bits))


def fp16_round_up(x: float) -> int:
    return int(lib().orc_fp16_round_up(float(x)))


def round_to_dtype_bits(x: float, dtype: str) -> int:
    L = lib()
    f = L.orc_bf16_from_double_rne if _is_bf16(dtype) else L.orc_fp16_from_double_rne
    return int(f(float(x)))


def dequant(code: int, scale_bits: int) -> float:
    return lib().orc_dequant(int(code), int(scale_bits))


# -------------------------------------------------------------- quantizer ---
def token_scale(row_bits: np.ndarray, dtype: str) -> int:
    row = np.ascontiguousarray(row_bits, dtype=np.uint16)
    return int(lib().orc_token_scale(_p(row), row.shape[-1], _is_bf16(dtype)))


def quantize_row(row_bits: np.ndarray, dtype: str, scale_bits: int) -> np.ndarray:
    row = np.ascontiguousarray(row_bits, dtype=np.uint16)
    out = np.empty(row.shape[-1], dtype=np.int8)
    lib().orc_quantize_row(_p(row), row.shape[-1], _is_bf16(dtype), int(scale_bits), _p(out))
    return out


def quantize_rows(x_bits: np.ndarray, dtype: str):
    """Rows [..., D] -> (codes int8 [..., D], scale bits uint16 [...])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    D = x.shape[-1]
    N = x.size // D if D else 0
    q = np.empty(x.shape, dtype=np.int8)
    s = np.empty(x.shape[:-1], dtype=np.uint16)
    lib().orc_quantize_rows(_p(x), N, D, _is_bf16(dtype), _p(q), _p(s))
    return q, s


def quantize_rows_static(x_bits: np.ndarray, dtype: str, scale: float) -> np.ndarray:
    """Static per-tensor scale (binary32): codes = clamp(rne(fl32(x * fl32(1/s))),
    +-127) ("fix: #552 int8 kv cache quantization cannot be enabled" (InfiniLM
    PR #553); "Add calibrated INT8 KV cache to PyTorch backend" (TensorRT-LLM
    PR #18953))."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    D = x.shape[-1]
    q = np.empty(x.shape, dtype=np.int8)
    lib().orc_quantize_rows_static(_p(x), x.size // D if D else 0, D, _is_bf16(dtype),
                                   float(np.float32(scale)), _p(q))
    return q


def prefill_sequence(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, dtype: str,
                     sm_scale: float, quantized: bool = True):
    """Causal attention of a chunk's n query tokens [n, Hq, D] (the last n of
    the sequence's L tokens k/v [L, Hkv, D]) over tokens 0..L-n+i ("fix(cuda/kv):
    correct Int8 KV per-token scale ..." (mlxcel PR #717), "Server integration":
    Int8 chunked prefill).  Returns (out float64 [n, Hq, D], out_bits)."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    n, Hq, D = q.shape
    L, Hkv, _ = k.shape
    if n > L or Hq % Hkv:
        raise ValueError("need n <= L and Hq a multiple of Hkv")
    out = np.empty((n, Hq, D), dtype=np.float64)
    out_bits = np.empty((n, Hq, D), dtype=np.uint16)
    work = np.empty(2 * max(L, 1) * D, dtype=np.float64)
    qwork = np.empty(D, dtype=np.int8)
    lib().orc_prefill_sequence(_p(q), _p(k), _p(v), L, n, Hq, Hkv, D, _is_bf16(dtype),
                               int(bool(quantized)), float(sm_scale), _p(out), _p(out_bits),
                               _p(work), _p(qwork))
    return out, out_bits


def trim_keep_sink(rows: np.ndarray, keep: int, n: int) -> np.ndarray:
    """Front trim keeping the first ``keep`` tokens: rows [L, ...] -> [L', ...]
    without the n tokens after the sink ("fix(cuda/kv): correct Int8 KV
    per-token scale ..." (mlxcel PR #717) follow-up, "The fix")."""
    a = np.ascontiguousarray(rows)
    L = a.shape[0]
    rb = a.nbytes // L if L else 0
    out = np.empty_like(a)
    m = lib().orc_trim_keep_sink(_p(a), L, rb, int(keep), int(n), _p(out))
    return out[:m]


def dequantize_rows(codes: np.ndarray, scales: np.ndarray, dtype: str) -> np.ndarray:
    """Codes [..., D] int8 times their row's FP16 scale [...], rounded (RNE)
    to ``dtype``: the dequantize-window baseline ("fix(cuda/kv): correct Int8
    KV per-token scale ..." (mlxcel PR #717), "The Int8 bug and fix")."""
    c = np.ascontiguousarray(codes, dtype=np.int8)
    sc = np.ascontiguousarray(scales, dtype=np.uint16).reshape(-1)
    D = c.shape[-1]
    assert c.size == sc.size * D
    out = np.empty(c.shape, dtype=np.uint16)
    lib().orc_dequantize_rows(_p(c), _p(sc), sc.size, D, _is_bf16(dtype), _p(out))
    return out


def quantize_append(k_bits, v_bits, dtype, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                    block_size: int) -> int:
    """Quantize-on-write of tokens [T, Hkv, D] into numpy cache arrays
    ([NB, Hkv, bs, D] int8 and [NB, Hkv, bs] uint16), in place.
    Returns the number of out-of-range slots (those tokens are not written)."""
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hkv, D = k.shape
    NB = k_cache.shape[0]
    for a, dt in ((k_cache, np.int8), (v_cache, np.int8), (k_scale, np.uint16),
                  (v_scale, np.uint16)):
        if a.dtype != dt or not a.flags.c_contiguous:
            raise ValueError("cache arrays must be C-contiguous with the right dtype")
    return int(lib().orc_quantize_append(_p(k), _p(v), Hkv * D, Hkv * D, T, Hkv, D,
                                         _is_bf16(dtype), _p(sm), _p(k_cache), _p(v_cache),
                                         _p(k_scale), _p(v_scale), NB, block_size))


# -------------------------------------------------------------- attention ---
def attend_one(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, sm_scale: float,
               partition: int | None = None) -> np.ndarray:
    """softmax(sm_scale * q . k_hat^T) v_hat for float64 q [D], k_hat/v_hat [L, D];
    with ``partition`` the log-sum-exp partitioned formulation is used."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k_hat, dtype=np.float64)
    v = np.ascontiguousarray(v_hat, dtype=np.float64)
    L, D = k.shape
    out = np.empty(D, dtype=np.float64)
    if partition is None:
        lib().orc_attend_one(_p(q), _p(k), _p(v), L, D, D, float(sm_scale), _p(out))
    else:
        scratch = np.empty(D, dtype=np.float64)
        lib().orc_attend_one_partitioned(_p(q), _p(k), _p(v), L, D, D, float(sm_scale),
                                         int(partition), _p(out), _p(scratch))
    return out


def decode_sequence(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, dtype: str,
                    sm_scale: float, quantized: bool = True, heads=None):
    """Decode of one sequence from its own token arrays.

    q_bits [Hq, D]; k_bits, v_bits [L, Hkv, D] (16-bit patterns as written).
    quantized=True: tokenwise INT8 quantize + dequantize first (the INT8 path);
    quantized=False: native 16-bit K/V (the reference for the 16-bit twin).
    Returns (out float64 [n, D], out_bits uint16 [n, D]) for the requested
    heads (all Hq by default)."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    Hq, D = q.shape
    L, Hkv, _ = k.shape
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    hl = None if heads is None else np.ascontiguousarray(heads, dtype=np.int32)
    n = Hq if hl is None else len(hl)
    out = np.empty((n, D), dtype=np.float64)
    out_bits = np.empty((n, D), dtype=np.uint16)
    work = np.empty(2 * max(L, 1) * D, dtype=np.float64)
    qwork = np.empty(D, dtype=np.int8)
    lib().orc_decode_sequence(_p(q), _p(k), _p(v), L, Hq, Hkv, D, _is_bf16(dtype),
                              int(bool(quantized)), float(sm_scale),
                              None if hl is None else _p(hl), n, _p(out), _p(out_bits),
                              _p(work), _p(qwork))
    return out, out_bits


def page_bytes_int8(block_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().orc_page_bytes_int8(block_size, num_kv_heads, head_dim))


def page_bytes_native16(block_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().orc_page_bytes_native16(block_size, num_kv_heads, head_dim))
