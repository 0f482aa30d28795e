"""The allocation-free decode entry point (kvq_paged_decode_noalloc).

It serves callers that may not allocate device memory themselves or let a
library do it: hosts that hand out all device memory from their own pool
(inference servers, framework plugins), programs with a memory budget fixed
at start-up, and latency-critical loops that must not risk the device-wide
synchronization cudaMalloc/cudaFree can cause.  Instead of a caller-provided
workspace it uses a fixed scratch array built into the library.

Checked here through the C ABI: on a workload whose long sequences go through
the split-K path (so the scratch is really used), two calls in a row match the
regular entry point within the tests' attention tolerance; sizes whose
workspace exceeds the built-in scratch are rejected with a clear status.  This
file is collected last so that a failure here never hides another test.
"""
import ctypes

import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import workloads as W
from _harness import Case, assert_attention_close, bits_f64, out_bits

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p
SCRATCH_LIMIT = 16 << 20      # KVQ_NOALLOC_SCRATCH_BYTES in include/kvq.h


def _noalloc(case: Case, out: torch.Tensor, max_ctx=None) -> int:
    w = case.w
    kc, vc, ks, vs = case.int8
    L = kvq.load()
    return L.kvq_paged_decode_noalloc(
        P(case.q.data_ptr()), 1 if w.dtype == "bf16" else 0, w.num_seqs, w.num_q_heads,
        w.num_kv_heads, w.head_dim, P(kc.data_ptr()), P(vc.data_ptr()), P(ks.data_ptr()),
        P(vs.data_ptr()), case.nb, 16, P(case.bt.data_ptr()), case.bt.shape[1],
        P(case.cl.data_ptr()), w.max_context_len if max_ctx is None else max_ctx, w.sm_scale,
        P(out.data_ptr()), P(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice():
    w = W.make("canonical")
    case = Case(w)
    case.write_prefix()
    case.write_step()
    need = kvq.kvq_decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                          w.head_dim, w.max_context_len)
    assert 0 < need <= SCRATCH_LIMIT          # split-K path: the scratch is used
    ref = out_bits(case.decode())
    for _ in range(2):                        # two calls in a row share the scratch
        out = torch.full_like(case.q, float("nan"))
        assert _noalloc(case, out) == 0
        torch.cuda.synchronize()
        got = out_bits(out)
        for b in range(w.num_seqs):
            assert_attention_close(got[b], bits_f64(ref[b], w.dtype), w.dtype, f"seq {b}")
    assert kvq.kvq_get_error() == (0, 0)


def test_noalloc_rejects_sizes_beyond_scratch():
    w = W.custom(2, 8, 1, 128, "bf16", [40, 40], seed=21)
    case = Case(w)
    out = torch.empty_like(case.q)
    L = kvq.load()
    # 256 sequences of 16K tokens with 64/8 heads need far more than the scratch
    big = kvq.kvq_decode_workspace_bytes(256, 64, 8, 128, 16384)
    assert big > SCRATCH_LIMIT
    st = L.kvq_paged_decode_noalloc(P(case.q.data_ptr()), 1, 256, 64, 8, 128, P(0), P(0), P(0),
                                    P(0), 1, 16, P(0), 1024, P(0), 16384, 0.1,
                                    P(out.data_ptr()), None)
    assert st == 4                            # KVQ_ERR_WORKSPACE_TOO_SMALL, nothing launched
    torch.cuda.synchronize()
