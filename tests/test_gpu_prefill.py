"""Chunked-prefill attention over the INT8 cache ("fix(cuda/kv): correct Int8
KV per-token scale ..." (mlxcel PR #717), "Server integration": Int8 chunked
prefill + decode over the same cache) through the C ABI, against the oracle's
causal attention over the dequantized tokens: every query row of every
sequence, for chunks from 0 tokens to the whole sequence, G in {1,2,3,4,8},
both head dims and activation dtypes; a one-query chunk equals the decode."""
import numpy as np
import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import oracle
import workloads as W
from _harness import Case, assert_attention_close, bits_f64, out_bits, to_dev

pytestmark = pytest.mark.gpu

LENS = [1, 17, 100, 300, 1000, 64, 40]
CHUNKS = [1, 17, 37, 64, 257, 0, 40]


def _queries(w, chunks, seed):
    r = np.random.default_rng(seed)
    x = r.standard_normal((sum(chunks), w.num_q_heads, w.head_dim)).astype(np.float32)
    if w.dtype == "fp16":
        return x.astype(np.float16).view(np.uint16)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(8, 2, 128, "bf16"), (4, 4, 64, "fp16"),
                                            (12, 4, 128, "fp16"), (16, 2, 64, "bf16"),
                                            (6, 3, 128, "bf16"), (4, 2, 64, "fp16")])
def test_prefill_matches_oracle(Hq, Hkv, D, dtype):
    w = W.custom(len(LENS), Hq, Hkv, D, dtype, LENS, seed=81 + Hq + D)
    case = Case(w)
    case.write_prefix()
    qb = _queries(w, CHUNKS, seed=Hq * 3 + D)
    qs = torch.tensor(np.concatenate([[0], np.cumsum(CHUNKS)]), dtype=torch.int32, device="cuda")
    q = to_dev(qb, dtype)
    out = kvq.kvq_paged_prefill(q, *case.int8, case.bt, case.cl, qs, w.max_context_len,
                                max(CHUNKS), w.sm_scale)
    ob = out_bits(out)
    start = 0
    for b, (L, n) in enumerate(zip(LENS, CHUNKS)):
        if n:
            k, v = w.seq_kv(b)
            ref, _ = oracle.prefill_sequence(qb[start:start + n], k, v, dtype, w.sm_scale)
            for i in range(n):
                assert_attention_close(ob[start + i], ref[i], dtype, f"seq {b} query {i}")
        start += n
    assert kvq.kvq_get_error() == (0, 0)


def test_one_query_chunk_equals_decode():
    w = W.custom(4, 8, 2, 128, "bf16", [33, 129, 700, 16], seed=89)
    case = Case(w)
    case.write_prefix()
    qs = torch.arange(5, dtype=torch.int32, device="cuda")
    out_p = kvq.kvq_paged_prefill(case.q.reshape(4, 8, 128), *case.int8, case.bt, case.cl, qs,
                                  w.max_context_len, 1, w.sm_scale)
    out_d = kvq.kvq_paged_decode(case.q, *case.int8, case.bt, case.cl, w.max_context_len,
                                 w.sm_scale)
    for b in range(4):
        ref, _ = oracle.decode_sequence(w.seq_q(b), *w.seq_kv(b), "bf16", w.sm_scale)
        assert_attention_close(out_bits(out_p)[b], ref, "bf16", f"prefill seq {b}")
        assert_attention_close(out_bits(out_d)[b], ref, "bf16", f"decode seq {b}")
    assert kvq.kvq_get_error() == (0, 0)


def test_prefill_flags_chunk_longer_than_context():
    w = W.custom(2, 4, 2, 64, "fp16", [10, 20], seed=91)
    case = Case(w)
    case.write_prefix()
    qs = torch.tensor([0, 12, 14], dtype=torch.int32, device="cuda")   # 12 > L = 10
    q = torch.zeros((14, 4, 64), dtype=torch.float16, device="cuda")
    kvq.kvq_paged_prefill(q, *case.int8, case.bt, case.cl, qs, w.max_context_len, 12, w.sm_scale)
    st, flags = kvq.kvq_get_error()
    assert st == 5 and flags & kvq.DEVERR_CONTEXT
    assert kvq.kvq_get_error() == (0, 0)


@pytest.mark.slow
def test_prefill_full_size_sampled():
    """The timed 8K shape (one sequence of 8192 cached tokens, all of them
    queries, 64 query / 8 KV heads, bf16) in the launch configuration the
    bench times; sampled query rows (both ends, tile and CTA boundaries, and
    random ones) against the oracle's decode over the row's causal prefix (a
    one-query chunk at position p is the decode over tokens 0..p)."""
    L, Hq, Hkv, D = 8192, 64, 8, 128
    w = W.custom(1, Hq, Hkv, D, "bf16", [L], seed=97)
    case = Case(w)
    case.write_prefix()
    qb = _queries(w, [L], seed=98)
    qs = torch.tensor([0, L], dtype=torch.int32, device="cuda")
    out = kvq.kvq_paged_prefill(to_dev(qb, "bf16"), *case.int8, case.bt, case.cl, qs, L, L,
                                w.sm_scale)
    ob = out_bits(out)
    k, v = w.seq_kv(0)
    rows = {0, 1, 15, 16, 31, 32, 63, 64, 4095, 4096, 8190, 8191}
    rows |= set(np.random.default_rng(99).integers(0, L, 12).tolist())
    for i in sorted(rows):
        ref, _ = oracle.decode_sequence(qb[i], k[:i + 1], v[:i + 1], "bf16", w.sm_scale)
        assert_attention_close(ob[i], ref, "bf16", f"query {i}")
    assert kvq.kvq_get_error() == (0, 0)


def _ramped(w, b, gain, spike=None):
    """Sequence b's K with magnitudes growing along the sequence (token t
    scaled by 1 + gain t), so the scores of later tiles exceed a row's
    running maximum by far more than 2^8 and the kernels' rescale of O runs
    again and again; `spike` = (token, factor) multiplies one token's key."""
    k, v = w.seq_kv(b)
    kf = bits_f64(k, w.dtype)
    kf *= (1.0 + gain * np.arange(kf.shape[0]))[:, None, None]
    if spike is not None:
        kf[spike[0]] *= spike[1]
    return W.to_bits(kf.astype(np.float32), w.dtype), v


@pytest.mark.parametrize("G,dtype,chunk", [(4, "bf16", 700), (1, "fp16", 700), (8, "bf16", 130)])
def test_prefill_rescale_path(G, dtype, chunk):
    """Scores that keep growing along the sequence (and one outsized key)
    drive the softmax's rescale of the TMEM accumulator: every row against
    the oracle (which has no such shortcut)."""
    Hkv, D, L = 2, 128, 700
    w = W.custom(2, G * Hkv, Hkv, D, dtype, [L, L], seed=101 + G)
    case = Case(w)
    seqs = [_ramped(w, 0, 0.02), _ramped(w, 1, 0.0, spike=(400, 40.0))]
    for b, (k, v) in enumerate(seqs):
        case._write(k, v, w.slots(b, 0, L))
    chunks = [chunk, chunk]
    qb = _queries(w, chunks, seed=102 + G)
    qs = torch.tensor([0, chunk, 2 * chunk], dtype=torch.int32, device="cuda")
    out = kvq.kvq_paged_prefill(to_dev(qb, dtype), *case.int8, case.bt, case.cl, qs, L, chunk,
                                w.sm_scale)
    ob = out_bits(out)
    for b, (k, v) in enumerate(seqs):
        ref, _ = oracle.prefill_sequence(qb[b * chunk:(b + 1) * chunk], k, v, dtype, w.sm_scale)
        for i in range(chunk):
            assert_attention_close(ob[b * chunk + i], ref[i], dtype, f"seq {b} query {i}")
    # the same caches through the decode (its running maximum moves every page)
    out_d = kvq.kvq_paged_decode(to_dev(qb[[chunk - 1, 2 * chunk - 1]], dtype), *case.int8,
                                 case.bt, case.cl, L, w.sm_scale)
    for b, (k, v) in enumerate(seqs):
        ref, _ = oracle.decode_sequence(qb[(b + 1) * chunk - 1], k, v, dtype, w.sm_scale)
        assert_attention_close(out_bits(out_d)[b], ref, dtype, f"decode seq {b}")
    assert kvq.kvq_get_error() == (0, 0)
