"""The dequantize-window baseline ("fix(cuda/kv): correct Int8 KV per-token
scale ..." (mlxcel PR #717), "The Int8 bug and fix": dequantize the cached
window, then attend over 16-bit values) through the C ABI.

* The window is bit-exact against the oracle (code * scale rounded once to the
  dtype) on every valid token of every sequence, read back through the block
  table, for ragged contexts and both head dims.
* The window followed by the 16-bit decode matches the oracle's native
  attention over the same rounded values (the twin's tolerance).
* Device-side checks: a block id out of range is flagged and skipped.
"""
import numpy as np
import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import oracle
import workloads as W
from _harness import BS, Case, assert_attention_close, out_bits, tdtype

pytestmark = pytest.mark.gpu

RAGGED = [0, 1, 15, 16, 17, 63, 250, 1000, 2049]


def _window_seq(case, kw, vw, b):
    """16-bit window values of sequence b read back through its block table."""
    L = int(case.w.context_lens[b])
    t = torch.arange(L, device="cuda")
    blk = case.bt[b, t // BS].long()
    off = t % BS
    f = lambda x: x[blk, :, off].cpu().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    return f(kw), f(vw)


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(8, 2, 128, "bf16"), (4, 4, 64, "fp16"),
                                            (12, 4, 128, "fp16")])
def test_window_bit_exact_and_attention(Hq, Hkv, D, dtype):
    w = W.custom(len(RAGGED), Hq, Hkv, D, dtype, RAGGED, seed=41 + D)
    case = Case(w)
    case.write_prefix()
    kw, vw = kvq.kvq_dequantize_window(*case.int8, case.bt, case.cl, w.max_context_len,
                                       tdtype(dtype))
    torch.cuda.synchronize()
    out = kvq.kvq_paged_decode_kv16(case.q, kw, vw, case.bt, case.cl, w.max_context_len,
                                    w.sm_scale)
    ob = out_bits(out)
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        k, v = w.seq_kv(b)
        qk, sk = oracle.quantize_rows(k, dtype)
        qv, sv = oracle.quantize_rows(v, dtype)
        want_k = oracle.dequantize_rows(qk, sk, dtype)
        want_v = oracle.dequantize_rows(qv, sv, dtype)
        got_k, got_v = _window_seq(case, kw, vw, b)
        assert np.array_equal(got_k, want_k[:L]), f"seq {b} K window"
        assert np.array_equal(got_v, want_v[:L]), f"seq {b} V window"
        ref, _ = oracle.decode_sequence(w.seq_q(b), want_k[:L], want_v[:L], dtype, w.sm_scale,
                                        quantized=False)
        assert_attention_close(ob[b], ref, dtype, f"window decode seq {b}")
    assert kvq.kvq_get_error() == (0, 0)


def test_window_flags_bad_block_and_skips_it():
    w = W.custom(2, 4, 2, 64, "fp16", [40, 40], seed=43)
    case = Case(w)
    case.write_prefix()
    bt = case.bt.clone()
    bt[1, 1] = case.nb + 5                       # out of range
    kw = torch.full((case.nb, 2, BS, 64), 7.0, dtype=torch.float16, device="cuda")
    vw = kw.clone()
    kvq.kvq_dequantize_window(*case.int8, bt, case.cl, w.max_context_len, torch.float16,
                              kw, vw)
    st, flags = kvq.kvq_get_error()
    assert st == 5 and flags & kvq.DEVERR_BLOCK
    # sequence 0 fully written; the bad page of sequence 1 left untouched
    k, _ = w.seq_kv(0)
    qk, sk = oracle.quantize_rows(k, "fp16")
    got0 = kw[case.bt[0, 0].long(), :, :].cpu().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got0.transpose(1, 0, 2), oracle.dequantize_rows(qk, sk, "fp16")[:BS])
    assert kvq.kvq_get_error() == (0, 0)
