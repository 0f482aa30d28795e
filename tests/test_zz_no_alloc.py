"""The allocation-free decode entry point (kvq_paged_decode_noalloc).

It serves callers that may not allocate device memory themselves or let a
library do it: hosts that hand out all device memory from their own pool
(inference servers, framework plugins), programs with a memory budget fixed
at start-up, and latency-critical loops that must not risk the device-wide
synchronization cudaMalloc/cudaFree can cause.  Instead of a caller-provided
workspace it uses a fixed scratch array built into the library
(KVQ_NOALLOC_SCRATCH_BYTES), handed to the regular launcher as its workspace.

Checked here through the C ABI:
* two calls in a row on the canonical workload equal the regular entry point
  bit for bit (same launcher decisions) and every (sequence, head) matches
  the oracle;
* the long-context workload, whose partials go through the scratch, then a
  different shape, then the long workload again: stale contents of the shared
  array never show;
* the serving mix (G = 8, D = 128), for which the recommended workspace is
  larger than the scratch: the launcher fits fewer ranges into it and the
  results equal the regular entry point given a workspace of the same size;
* a shape for which not even one range per KV head fits is refused.
This file is collected last so that a failure here never hides another test.
"""
import ctypes

import numpy as np
import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import oracle
import workloads as W
from _harness import Case, assert_attention_close, out_bits

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p
SCRATCH_LIMIT = 16 << 20      # KVQ_NOALLOC_SCRATCH_BYTES in include/kvq.h


def _noalloc(case: Case, out: torch.Tensor) -> int:
    w = case.w
    kc, vc, ks, vs = case.int8
    L = kvq.load()
    return L.kvq_paged_decode_noalloc(
        P(case.q.data_ptr()), 1 if w.dtype == "bf16" else 0, w.num_seqs, w.num_q_heads,
        w.num_kv_heads, w.head_dim, P(kc.data_ptr()), P(vc.data_ptr()), P(ks.data_ptr()),
        P(vs.data_ptr()), case.nb, 16, P(case.bt.data_ptr()), case.bt.shape[1],
        P(case.cl.data_ptr()), w.max_context_len, w.sm_scale, P(out.data_ptr()),
        P(torch.cuda.current_stream().cuda_stream))


def _run(case: Case) -> np.ndarray:
    out = torch.full_like(case.q, float("nan"))
    assert _noalloc(case, out) == 0
    torch.cuda.synchronize()
    return out_bits(out)


def _regular(case: Case, ws_bytes=None) -> np.ndarray:
    """kvq_paged_decode with the recommended workspace, or one of ws_bytes."""
    ws = None
    if ws_bytes is not None:
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    return out_bits(case.decode() if ws is None else
                    kvq.kvq_paged_decode(case.q, *case.int8, case.bt, case.cl,
                                         case.w.max_context_len, case.w.sm_scale, workspace=ws))


def _resident(name_or_w) -> Case:
    w = W.make(name_or_w) if isinstance(name_or_w, str) else name_or_w
    case = Case(w)
    case.write_prefix()
    case.write_step()
    return case


def _oracle_pairs(case: Case, got: np.ndarray, seqs, heads_per_seq=4, seed=0):
    w = case.w
    r = np.random.default_rng(seed)
    for b in seqs:
        heads = sorted(r.choice(w.num_q_heads, size=min(heads_per_seq, w.num_q_heads),
                                replace=False))
        ref, _ = oracle.decode_sequence(w.seq_q(b), *w.seq_kv(b), w.dtype, w.sm_scale,
                                        heads=heads)
        assert_attention_close(got[b, heads], ref, w.dtype, f"seq {b} heads {heads}")


def _need(w) -> int:
    return kvq.kvq_decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                          w.head_dim, w.max_context_len)


def test_noalloc_equals_workspace_entry_point_twice():
    case = _resident("canonical")
    w = case.w
    assert 0 < _need(w) <= SCRATCH_LIMIT      # split-K with the same ranges as the regular call
    ref = _regular(case)
    for _ in range(2):                        # two calls in a row share the scratch
        got = _run(case)
        assert np.array_equal(got, ref)
    _oracle_pairs(case, got, range(w.num_seqs), heads_per_seq=w.num_q_heads)
    assert kvq.kvq_get_error() == (0, 0)


@pytest.mark.slow
def test_noalloc_long_context_then_another_shape_then_long_again():
    long_case = _resident("long")
    assert 0 < _need(long_case.w) <= SCRATCH_LIMIT
    ref_long = _regular(long_case)
    got = _run(long_case)
    assert np.array_equal(got, ref_long)
    _oracle_pairs(long_case, got, range(4), seed=1)
    # a different shape (G = 8, ragged, D = 64) through the same array
    other = _resident(W.custom(9, 16, 2, 64, "bf16", [1, 17, 250, 4100, 33, 2000, 64, 999, 3],
                               seed=71))
    got_o = _run(other)
    assert np.array_equal(got_o, _regular(other))
    _oracle_pairs(other, got_o, range(9), heads_per_seq=16, seed=2)
    # the first shape again: nothing of the second call's partials leaks in
    assert np.array_equal(_run(long_case), ref_long)
    assert kvq.kvq_get_error() == (0, 0)


@pytest.mark.slow
def test_noalloc_serving_mix_beyond_the_recommended_workspace():
    case = _resident("serving")
    w = case.w
    assert _need(w) > SCRATCH_LIMIT           # G = 8, D = 128: fewer ranges than recommended
    got = _run(case)
    assert np.array_equal(got, _regular(case, SCRATCH_LIMIT))
    L = w.context_lens
    seqs = {int(np.argmax(L)), int(np.argmin(L))}
    seqs |= set(np.random.default_rng(3).choice(w.num_seqs, 4, replace=False).tolist())
    _oracle_pairs(case, got, sorted(seqs), seed=4)
    assert kvq.kvq_get_error() == (0, 0)


def test_noalloc_refuses_shapes_without_one_range_per_kv_head():
    """8 (G) x 2100 KV heads at D = 128 need 2100 ranges of 8,256 bytes
    (17.3 MB) even at one range per KV head: refused before anything runs
    (the small tensors below are never read).  The context bound (1024
    tokens, 64 pages) is past the no-split limit of four pages, so the call
    takes the split path that needs the scratch."""
    L = kvq.load()
    x = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    p = P(x.data_ptr())
    Hkv, G = 2100, 8
    st = L.kvq_paged_decode_noalloc(p, 1, 1, G * Hkv, Hkv, 128, p, p, p, p, 64, 16, p, 64, p,
                                    1024, 0.1, p, None)
    assert st == 4                            # KVQ_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert kvq.kvq_get_error() == (0, 0)
