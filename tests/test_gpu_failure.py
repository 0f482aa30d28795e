"""Failure detection without a GPU fault: a device-side wait that nothing
completes gives up after its limit, the kernel reports KVQ_DEVERR_TIMEOUT
through the error word, kvq_get_error returns KVQ_ERR_DEVICE_TIMEOUT and
clears it, and the context stays usable (a decode right after is correct)."""
import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import workloads as W
from _harness import Case, assert_attention_close, out_bits
import oracle

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    assert kvq.kvq_get_error() == (0, 0)
    kvq.kvq_selftest_wait_timeout(2000)                  # 2 ms
    st, flags = kvq.kvq_get_error()
    assert st == 6 and flags == kvq.DEVERR_TIMEOUT
    assert kvq.kvq_get_error() == (0, 0)                 # cleared
    w = W.make("tiny")
    case = Case(w)
    case.write_prefix()
    ob = out_bits(case.decode())
    for b in range(w.num_seqs):
        ref, _ = oracle.decode_sequence(w.seq_q(b), *w.seq_kv(b), w.dtype, w.sm_scale)
        assert_attention_close(ob[b], ref, w.dtype, f"decode after timeout seq {b}")
    assert kvq.kvq_get_error() == (0, 0)


def test_selftest_rejects_bad_limits():
    for bad in (0, 1000001):
        with pytest.raises(kvq.KvqError):
            kvq.kvq_selftest_wait_timeout(bad)
