"""Python binding of libkvq: tokenwise symmetric INT8 paged KV cache for decode.

Argument marshalling only.  Every step of the hot path runs in the CUDA
kernels of ``libkvq.so`` (built in-tree for sm_103a by ``_build.build()``);
there is no Python or CPU implementation of any operation here, and a missing
library is an error, not a fallback.

The functions mirror the C ABI in ``include/kvq.h`` (same names) and take
torch CUDA tensors, passing their device pointers and the current CUDA
stream:

* ``kvq_quantize_append``  -- quantize-on-write of new K/V rows into the
  paged INT8 cache ("feat: opt-in INT8 KV-cache quantization", MoE-Infinity
  PR #183, "What landed"; "fix(cuda/kv): correct Int8 KV per-token scale",
  mlxcel PR #717, "The Int8 bug and fix").
* ``kvq_paged_decode``     -- fused paged decode attention over INT8 K/V.
* ``kvq_paged_decode_kv16`` / ``kvq_cache_append_kv16`` -- the native 16-bit
  twin used for A/B comparison.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

from . import _build

__all__ = [
    "KvqError", "load", "kvq_quantize_append", "kvq_paged_decode", "kvq_paged_decode_kv16",
    "kvq_cache_append_kv16", "kvq_paged_decode_noalloc", "kvq_dequantize_window",
    "kvq_quantize_append_static", "kvq_paged_decode_static", "kvq_trim_front_keep_sink",
    "kvq_paged_prefill", "kvq_selftest_wait_timeout", "kvq_paged_decode_cuda_cores",
    "kvq_decode_workspace_bytes", "kvq_decode_partition_pages",
    "kvq_get_error", "kvq_status_string", "alloc_int8_cache", "alloc_kv16_cache",
    "HEADER_SYMBOLS", "BLOCK_SIZE", "DEVERR_SLOT", "DEVERR_BLOCK", "DEVERR_CONTEXT",
    "DEVERR_TIMEOUT",
]

BLOCK_SIZE = 16
FP16, BF16 = 0, 1
DEVERR_SLOT, DEVERR_BLOCK, DEVERR_CONTEXT, DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8
STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARGUMENT", 2: "KVQ_ERR_UNSUPPORTED",
          3: "KVQ_ERR_CUDA", 4: "KVQ_ERR_WORKSPACE_TOO_SMALL", 5: "KVQ_ERR_DEVICE_INDEX",
          6: "KVQ_ERR_DEVICE_TIMEOUT"}

# Every function include/kvq.h declares (checked against the library's exports).
HEADER_SYMBOLS = (
    "kvq_quantize_append", "kvq_paged_decode", "kvq_decode_workspace_bytes",
    "kvq_decode_partition_pages", "kvq_paged_decode_split", "kvq_decode_workspace_bytes_split",
    "kvq_paged_decode_kv16", "kvq_paged_decode_kv16_split", "kvq_cache_append_kv16",
    "kvq_get_error", "kvq_status_string", "kvq_version", "kvq_paged_decode_noalloc",
    "kvq_dequantize_window", "kvq_quantize_append_static", "kvq_paged_decode_static",
    "kvq_trim_front_keep_sink", "kvq_paged_prefill", "kvq_selftest_wait_timeout",
    "kvq_paged_decode_cuda_cores",
)

_lib = None
LIB_PATH = _build.LIB


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libkvq.so (building it first if absent and nvcc exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not LIB_PATH.exists() or not _build.up_to_date():
        if not build_if_missing:
            raise RuntimeError(f"{LIB_PATH} is missing or stale; run _build.build()")
        _build.build()
    L = ctypes.CDLL(str(LIB_PATH))
    vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                             ctypes.c_size_t)
    L.kvq_quantize_append.argtypes = [vp, vp, i64, i64, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                      i32, i32, vp]
    L.kvq_cache_append_kv16.argtypes = [vp, vp, i64, i64, i32, i32, i32, i32, vp, vp, vp, i32,
                                        i32, vp]
    dec = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, i32, i32, vp, i32, vp, i32, f32, vp, vp,
           sz]
    L.kvq_paged_decode.argtypes = dec + [vp]
    L.kvq_paged_decode_split.argtypes = dec + [i32, vp]
    L.kvq_paged_decode_cuda_cores.argtypes = dec + [vp]
    L.kvq_paged_decode_noalloc.argtypes = dec[:-2] + [vp]
    L.kvq_paged_decode_noalloc.restype = ctypes.c_int
    dec16 = [vp, i32, i32, i32, i32, i32, vp, vp, i32, i32, vp, i32, vp, i32, f32, vp, vp, sz]
    L.kvq_paged_decode_kv16.argtypes = dec16 + [vp]
    L.kvq_paged_decode_kv16_split.argtypes = dec16 + [i32, vp]
    L.kvq_dequantize_window.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, i32, i32, vp,
                                        i32, i32, vp, vp, vp]
    f32s = ctypes.c_float
    L.kvq_paged_prefill.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, i32, i32, vp,
                                    i32, vp, i32, vp, i32, i32, f32s, vp, vp]
    L.kvq_trim_front_keep_sink.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, i32, i32, vp,
                                           vp, i32, vp]
    L.kvq_quantize_append_static.argtypes = [vp, vp, i64, i64, i32, i32, i32, i32, vp, vp, vp,
                                             f32s, f32s, i32, i32, vp]
    L.kvq_paged_decode_static.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp, f32s, f32s, i32,
                                          i32, vp, i32, vp, i32, f32s, vp, vp, sz, vp]
    for fn in ("kvq_quantize_append", "kvq_cache_append_kv16", "kvq_paged_decode",
               "kvq_paged_decode_cuda_cores",
               "kvq_paged_decode_split", "kvq_paged_decode_kv16", "kvq_paged_decode_kv16_split",
               "kvq_dequantize_window", "kvq_quantize_append_static", "kvq_paged_decode_static",
               "kvq_trim_front_keep_sink", "kvq_paged_prefill"):
        getattr(L, fn).restype = ctypes.c_int
    L.kvq_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.kvq_decode_workspace_bytes.restype = sz
    L.kvq_decode_workspace_bytes_split.argtypes = [i32, i32, i32, i32, i32, i32]
    L.kvq_decode_workspace_bytes_split.restype = sz
    L.kvq_decode_partition_pages.argtypes = [i32, i32, i32, i32, i32]
    L.kvq_decode_partition_pages.restype = i32
    L.kvq_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
    L.kvq_selftest_wait_timeout.restype = ctypes.c_int
    L.kvq_get_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    L.kvq_get_error.restype = ctypes.c_int
    L.kvq_status_string.argtypes = [ctypes.c_int]
    L.kvq_status_string.restype = ctypes.c_char_p
    L.kvq_version.argtypes = []
    L.kvq_version.restype = i32
    _lib = L
    return L


# ----------------------------------------------------------------- helpers ---
def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return FP16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"activations must be float16 or bfloat16, got {t.dtype}")


def _ptr(t):
    return None if t is None else t.data_ptr()     # an int; the argtypes make it a void*


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device=None):
    """The stream handle to launch on: `stream`, else the current stream of
    `device` (a torch.device of a CUDA tensor), else of the current device."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        idx = device.index if device is not None and device.index is not None else \
            torch.cuda.current_device()
        return _raw_stream(idx)
    return torch.cuda.current_stream(device).cuda_stream


def _check(status: int, what: str):
    if status != 0:
        raise KvqError(status, what)


def _rows(x: torch.Tensor, name: str):
    if x.dim() != 3 or x.stride(2) != 1 or (x.shape[1] > 1 and x.stride(1) != x.shape[2]):
        raise ValueError(f"{name} must be [T, Hkv, D] with contiguous heads")
    return x.stride(0)


def _need(cond: bool, msg: str):
    if not cond:
        raise ValueError(msg)


def _check_cache(kc, vc, Hkv, D, dtypes, name="cache"):
    _need(kc.is_cuda and vc.is_cuda, f"{name} must be CUDA tensors")
    _need(kc.dim() == 4 and kc.shape[1:] == (Hkv, BLOCK_SIZE, D) and vc.shape == kc.shape,
          f"{name} must be [num_blocks, {Hkv}, {BLOCK_SIZE}, {D}], got {tuple(kc.shape)}")
    _need(kc.dtype in dtypes and vc.dtype == kc.dtype, f"{name} dtype {kc.dtype}")
    _need(kc.is_contiguous() and vc.is_contiguous(), f"{name} must be contiguous")


def _check_scales(ks, vs, kc):
    _need(ks.shape == kc.shape[:3] and vs.shape == ks.shape, "scale planes must be [NB, Hkv, 16]")
    _need(ks.dtype in (torch.int16, torch.uint16) and vs.dtype == ks.dtype,
          "scale planes hold FP16 bits as int16")
    _need(ks.is_contiguous() and vs.is_contiguous(), "scale planes must be contiguous")


def _check_rows(k, v, slot_mapping):
    _need(k.is_cuda and v.is_cuda and slot_mapping.is_cuda, "inputs must be CUDA tensors")
    _need(k.shape == v.shape and k.dtype == v.dtype, "k and v must match")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.shape == (k.shape[0],)
          and slot_mapping.is_contiguous(), "slot_mapping must be int64 [T]")


def alloc_int8_cache(num_blocks: int, num_kv_heads: int, head_dim: int, device="cuda"):
    """(k_cache, v_cache, k_scale, v_scale) in the library's layout: int8
    [NB, Hkv, 16, D] payloads and int16 (FP16 bits) [NB, Hkv, 16] scale planes,
    zero-filled."""
    kc = torch.zeros((num_blocks, num_kv_heads, BLOCK_SIZE, head_dim), dtype=torch.int8,
                     device=device)
    ks = torch.zeros((num_blocks, num_kv_heads, BLOCK_SIZE), dtype=torch.int16, device=device)
    return kc, torch.zeros_like(kc), ks, torch.zeros_like(ks)


def alloc_kv16_cache(num_blocks: int, num_kv_heads: int, head_dim: int, dtype, device="cuda"):
    kc = torch.zeros((num_blocks, num_kv_heads, BLOCK_SIZE, head_dim), dtype=dtype, device=device)
    return kc, torch.zeros_like(kc)


# ----------------------------------------------------------- entry points ---
def kvq_quantize_append(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, stream=None):
    """Quantize new rows k, v [T, Hkv, D] into the paged INT8 cache at
    slot_mapping [T] (int64; negative = skip)."""
    L = load()
    T, Hkv, D = k.shape
    _check_rows(k, v, slot_mapping)
    _check_cache(k_cache, v_cache, Hkv, D, (torch.int8,))
    _check_scales(k_scale, v_scale, k_cache)
    st = L.kvq_quantize_append(_ptr(k), _ptr(v), _rows(k, "k"), _rows(v, "v"), T, Hkv, D,
                               _dtype_code(k), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
                               _ptr(k_scale), _ptr(v_scale), k_cache.shape[0], k_cache.shape[2],
                               _stream(stream))
    _check(st, "kvq_quantize_append")


def kvq_quantize_append_static(k, v, slot_mapping, k_cache, v_cache, k_scale: float,
                               v_scale: float, stream=None):
    """Quantize-on-write with static per-tensor scales (binary32): codes only,
    code = clamp(rne(fl32(x * fl32(1/scale))), +-127)."""
    L = load()
    _check_cache(k_cache, v_cache, k_cache.shape[1], k_cache.shape[3], (torch.int8,))
    _check_rows(k, v, slot_mapping)
    st = L.kvq_quantize_append_static(_ptr(k), _ptr(v), _rows(k, "k"), _rows(v, "v"), k.shape[0],
                                      k.shape[1], k.shape[2], _dtype_code(k), _ptr(slot_mapping),
                                      _ptr(k_cache), _ptr(v_cache), float(k_scale),
                                      float(v_scale), k_cache.shape[0], k_cache.shape[2],
                                      _stream(stream))
    _check(st, "kvq_quantize_append_static")


def kvq_paged_decode_static(q, k_cache, v_cache, k_scale: float, v_scale: float, block_tables,
                            context_lens, max_context_len: int, sm_scale: float, out=None,
                            workspace=None, stream=None):
    """Paged decode over an INT8 cache with static per-tensor scales."""
    L = load()
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _check_decode(q, k_cache, v_cache, block_tables, context_lens, out, (torch.int8,))
    ws, nbytes = _workspace(q, Hkv, max_context_len, 0, workspace)
    st = L.kvq_paged_decode_static(_ptr(q), _dtype_code(q), B, Hq, Hkv, D, _ptr(k_cache),
                                   _ptr(v_cache), float(k_scale), float(v_scale), NB, bs,
                                   _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                   int(max_context_len), float(sm_scale), _ptr(out), _ptr(ws),
                                   nbytes, _stream(stream))
    _check(st, "kvq_paged_decode_static")
    return out


def kvq_cache_append_kv16(k, v, slot_mapping, k_cache, v_cache, stream=None):
    L = load()
    T, Hkv, D = k.shape
    _check_rows(k, v, slot_mapping)
    _check_cache(k_cache, v_cache, Hkv, D, (k.dtype,))
    st = L.kvq_cache_append_kv16(_ptr(k), _ptr(v), _rows(k, "k"), _rows(v, "v"), T, Hkv, D,
                                 _dtype_code(k), _ptr(slot_mapping), _ptr(k_cache),
                                 _ptr(v_cache), k_cache.shape[0], k_cache.shape[2],
                                 _stream(stream))
    _check(st, "kvq_cache_append_kv16")


def kvq_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len,
                               partition_pages: int = 0) -> int:
    L = load()
    if partition_pages:
        return int(L.kvq_decode_workspace_bytes_split(num_seqs, num_q_heads, num_kv_heads,
                                                      head_dim, max_context_len,
                                                      partition_pages))
    return int(L.kvq_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                            max_context_len))


def kvq_decode_partition_pages(num_seqs, num_q_heads, num_kv_heads, head_dim,
                               max_context_len) -> int:
    return int(load().kvq_decode_partition_pages(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 max_context_len))


def _check_decode(q, k_cache, v_cache, block_tables, context_lens, out, cache_dtypes):
    _need(q.is_cuda and q.dim() == 3 and q.is_contiguous(), "q must be contiguous [B, Hq, D]")
    B, Hq, D = q.shape
    _check_cache(k_cache, v_cache, k_cache.shape[1], D, cache_dtypes)
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2
          and block_tables.shape[0] == B and block_tables.is_contiguous(),
          "block_tables must be contiguous int32 [B, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.shape == (B,)
          and context_lens.is_contiguous(), "context_lens must be int32 [B]")
    _need(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(),
          "out must match q")


_ws_need = {}


def _workspace(q, Hkv, max_context_len, partition_pages, workspace):
    B, Hq, D = q.shape
    key = (B, Hq, Hkv, D, int(max_context_len), int(partition_pages))
    need = _ws_need.get(key)
    if need is None:
        need = kvq_decode_workspace_bytes(B, Hq, Hkv, D, max_context_len, partition_pages)
        if len(_ws_need) < 4096:
            _ws_need[key] = need
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return workspace, nbytes


def kvq_paged_decode(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                     max_context_len: int, sm_scale: float, out=None, workspace=None,
                     partition_pages: int = 0, stream=None):
    """Paged decode over the INT8 cache.  q [B, Hq, D]; block_tables int32
    [B, max_blocks]; context_lens int32 [B]; returns out [B, Hq, D].
    ``workspace``: None allocates kvq_decode_workspace_bytes; an empty tensor
    runs without split-K (one warp per (sequence, KV head)).
    ``partition_pages``: 0 = balanced work ranges; >= 1 forces the range
    length in pages."""
    L = load()
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _check_decode(q, k_cache, v_cache, block_tables, context_lens, out, (torch.int8,))
    _check_scales(k_scale, v_scale, k_cache)
    ws, nbytes = _workspace(q, Hkv, max_context_len, partition_pages, workspace)
    args = [_ptr(q), _dtype_code(q), B, Hq, Hkv, D, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
            _ptr(v_scale), NB, bs, _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
            int(max_context_len), float(sm_scale), _ptr(out), _ptr(ws), nbytes]
    if partition_pages:
        st = L.kvq_paged_decode_split(*args, int(partition_pages), _stream(stream))
    else:
        st = L.kvq_paged_decode(*args, _stream(stream))
    _check(st, "kvq_paged_decode")
    return out


def kvq_paged_decode_cuda_cores(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                context_lens, max_context_len: int, sm_scale: float, out=None,
                                workspace=None, stream=None):
    """kvq_paged_decode with the page math on the CUDA cores (FFMA) instead of
    the tensor cores: the A/B counterpart, same arguments and results."""
    L = load()
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _check_decode(q, k_cache, v_cache, block_tables, context_lens, out, (torch.int8,))
    _check_scales(k_scale, v_scale, k_cache)
    ws, nbytes = _workspace(q, Hkv, max_context_len, 0, workspace)
    st = L.kvq_paged_decode_cuda_cores(_ptr(q), _dtype_code(q), B, Hq, Hkv, D, _ptr(k_cache),
                                       _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), NB, bs,
                                       _ptr(block_tables), block_tables.shape[1],
                                       _ptr(context_lens), int(max_context_len),
                                       float(sm_scale), _ptr(out), _ptr(ws), nbytes,
                                       _stream(stream))
    _check(st, "kvq_paged_decode_cuda_cores")
    return out


def kvq_paged_decode_noalloc(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                             max_context_len: int, sm_scale: float, out, stream=None):
    """kvq_paged_decode without a workspace, for callers that cannot allocate
    device memory: the split-K scratch is a fixed array inside the library
    (KVQ_NOALLOC_SCRATCH_BYTES per GPU).  ``out`` must be given.  Calls that
    overlap on the GPU share that scratch and race."""
    L = load()
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    _check_decode(q, k_cache, v_cache, block_tables, context_lens, out, (torch.int8,))
    _check_scales(k_scale, v_scale, k_cache)
    st = L.kvq_paged_decode_noalloc(_ptr(q), _dtype_code(q), B, Hq, Hkv, D, _ptr(k_cache),
                                    _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), NB, bs,
                                    _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                    int(max_context_len), float(sm_scale), _ptr(out),
                                    _stream(stream))
    _check(st, "kvq_paged_decode_noalloc")
    return out


def kvq_paged_decode_kv16(q, k_cache, v_cache, block_tables, context_lens, max_context_len: int,
                          sm_scale: float, out=None, workspace=None, partition_pages: int = 0,
                          stream=None):
    """Paged decode over the native 16-bit cache (same dtype as q)."""
    L = load()
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _check_decode(q, k_cache, v_cache, block_tables, context_lens, out, (q.dtype,))
    ws, nbytes = _workspace(q, Hkv, max_context_len, partition_pages, workspace)
    args = [_ptr(q), _dtype_code(q), B, Hq, Hkv, D, _ptr(k_cache), _ptr(v_cache), NB, bs,
            _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), int(max_context_len),
            float(sm_scale), _ptr(out), _ptr(ws), nbytes]
    if partition_pages:
        st = L.kvq_paged_decode_kv16_split(*args, int(partition_pages), _stream(stream))
    else:
        st = L.kvq_paged_decode_kv16(*args, _stream(stream))
    _check(st, "kvq_paged_decode_kv16")
    return out


def kvq_dequantize_window(k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                          max_context_len: int, dtype, k_out=None, v_out=None, stream=None):
    """Dequantize-window baseline: writes s * code, rounded to ``dtype``
    (torch.float16 / torch.bfloat16), for every page the sequences reach into
    a 16-bit cache of the INT8 cache's layout; returns (k_out, v_out)."""
    L = load()
    NB, Hkv, bs, D = k_cache.shape
    _check_cache(k_cache, v_cache, Hkv, D, (torch.int8,))
    _check_scales(k_scale, v_scale, k_cache)
    _need(dtype in (torch.float16, torch.bfloat16), "dtype must be float16 or bfloat16")
    B = context_lens.shape[0]
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2
          and block_tables.shape[0] == B and block_tables.is_contiguous(),
          "block_tables must be contiguous int32 [B, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.is_contiguous(),
          "context_lens must be int32 [B]")
    if k_out is None:
        k_out, v_out = alloc_kv16_cache(NB, Hkv, D, dtype, k_cache.device)
    _check_cache(k_out, v_out, Hkv, D, (dtype,))
    _need(k_out.shape == k_cache.shape, "k_out/v_out must have the INT8 cache's shape")
    st = L.kvq_dequantize_window(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), NB,
                                 bs, Hkv, D, _ptr(block_tables), B, block_tables.shape[1],
                                 _ptr(context_lens), int(max_context_len),
                                 BF16 if dtype == torch.bfloat16 else FP16, _ptr(k_out),
                                 _ptr(v_out), _stream(stream))
    _check(st, "kvq_dequantize_window")
    return k_out, v_out


def kvq_trim_front_keep_sink(k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                             trim, keep: int, stream=None):
    """Front trim keeping the first ``keep`` tokens of each sequence: drops
    trim[b] tokens after them (payload and scales in lockstep) and updates
    context_lens in place.  k_scale/v_scale None for a static-scale cache."""
    L = load()
    NB, Hkv, bs, D = k_cache.shape
    _check_cache(k_cache, v_cache, Hkv, D, (torch.int8,))
    if k_scale is not None:
        _check_scales(k_scale, v_scale, k_cache)
    B = context_lens.shape[0]
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2
          and block_tables.shape[0] == B and block_tables.is_contiguous(),
          "block_tables must be contiguous int32 [B, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.is_contiguous(),
          "context_lens must be int32 [B]")
    _need(trim.dtype == torch.int32 and trim.shape == (B,) and trim.is_contiguous(),
          "trim must be int32 [B]")
    st = L.kvq_trim_front_keep_sink(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                    NB, bs, Hkv, D, _ptr(block_tables), B, block_tables.shape[1],
                                    _ptr(context_lens), _ptr(trim), int(keep), _stream(stream))
    _check(st, "kvq_trim_front_keep_sink")


def kvq_paged_prefill(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                      query_start, max_context_len: int, max_query_len: int, sm_scale: float,
                      out=None, stream=None):
    """Chunked-prefill attention over the INT8 cache.  q [total_q, Hq, D]: the
    queries of each sequence's last n_b = query_start[b+1] - query_start[b]
    tokens (already in the cache), attending causally; returns out like q."""
    L = load()
    _need(q.is_cuda and q.dim() == 3 and q.is_contiguous(), "q must be contiguous [T, Hq, D]")
    T, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    _check_cache(k_cache, v_cache, Hkv, D, (torch.int8,))
    _check_scales(k_scale, v_scale, k_cache)
    B = context_lens.shape[0]
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2
          and block_tables.shape[0] == B and block_tables.is_contiguous(),
          "block_tables must be contiguous int32 [B, max_blocks]")
    _need(context_lens.dtype == torch.int32 and context_lens.is_contiguous(),
          "context_lens must be int32 [B]")
    _need(query_start.dtype == torch.int32 and query_start.shape == (B + 1,)
          and query_start.is_contiguous(), "query_start must be int32 [B + 1]")
    if out is None:
        out = torch.empty_like(q)
    _need(out.shape == q.shape and out.dtype == q.dtype and out.is_contiguous(), "out must match q")
    st = L.kvq_paged_prefill(_ptr(q), _dtype_code(q), B, Hq, Hkv, D, _ptr(k_cache), _ptr(v_cache),
                             _ptr(k_scale), _ptr(v_scale), NB, bs, _ptr(block_tables),
                             block_tables.shape[1], _ptr(context_lens), int(max_context_len),
                             _ptr(query_start), T, int(max_query_len), float(sm_scale),
                             _ptr(out), _stream(stream))
    _check(st, "kvq_paged_prefill")
    return out


def kvq_selftest_wait_timeout(limit_us: int, stream=None):
    """Launch the bounded-wait self-test (a wait that nothing completes, given
    up after limit_us); read the result with kvq_get_error."""
    _check(load().kvq_selftest_wait_timeout(int(limit_us), _stream(stream)),
           "kvq_selftest_wait_timeout")


def kvq_get_error(stream=None):
    """Synchronize, read and clear the device error word: (status, flags)."""
    flags = ctypes.c_uint32(0)
    st = load().kvq_get_error(_stream(stream), ctypes.byref(flags))
    return int(st), int(flags.value)


def kvq_status_string(status: int) -> str:
    return load().kvq_status_string(int(status)).decode()
