"""The upper and lower ends of the input range, through the C ABI, against the
oracle.

"feat: opt-in INT8 KV-cache quantization" (MoE-Infinity PR #183), "What
landed", states the quantizer's contract for any row: an upward-rounded FP16
scale absmax/127, codes in [-127, 127], element error at most scale/2.  For
BF16 activations that holds up to absmax = 127 * 65504 (about 8.3e6), where
the FP16 scale saturates; for FP16 activations it holds over their whole
range.  The kernels must therefore stay finite and accurate far outside the
N(0, 1) values of the workloads:

* V rows whose absmax lies beyond 65504 (BF16) or at 65504 (FP16): the code
  times its scale is not an FP16 number there;
* BF16 queries beyond 65504 or below 2^-14 (outside FP16's normal range);
* in the chunked prefill, V scales above 256 while the softmax's lazily
  rescaled probabilities reach 2^8.

Values are the workloads' N(0, 1) draws times a power of two, so the codes
are those of the unscaled draw and the oracle's output scales by the same
factor; the absolute tolerance scales with it (attention is linear in V).
Queries scaled by 2^k come with sm_scale times 2^-k, which keeps the softmax
of the N(0, 1) case."""
import numpy as np
import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import oracle
import workloads as W
from _harness import Case, assert_attention_close, bits_f64, out_bits, to_dev

pytestmark = pytest.mark.gpu

LENS = [1, 16, 37, 300, 2000]


def _decode_vs_oracle(w, seqs, q_bits, sm_scale, v_scale=1.0, parts=(0, 4), what=""):
    """Write (k, v) bits per sequence, decode (balanced launcher and forced
    4-page ranges, so both whole-sequence and split-K paths run) and compare
    every (sequence, head) with the oracle."""
    case = Case(w)
    for b, (k, v) in enumerate(seqs):
        case._write(k, v, w.slots(b, 0, len(k)))
    q = to_dev(q_bits, w.dtype)
    refs = [oracle.decode_sequence(q_bits[b], k, v, w.dtype, sm_scale)[0]
            for b, (k, v) in enumerate(seqs)]
    for P in parts:
        ob = out_bits(kvq.kvq_paged_decode(q, *case.int8, case.bt, case.cl, w.max_context_len,
                                           sm_scale, partition_pages=P))
        for b in range(w.num_seqs):
            assert_attention_close(ob[b], refs[b], w.dtype, f"{what} P={P} seq {b}", v_scale)
    ob = out_bits(kvq.kvq_paged_decode_cuda_cores(q, *case.int8, case.bt, case.cl,
                                                  w.max_context_len, sm_scale))
    for b in range(w.num_seqs):
        assert_attention_close(ob[b], refs[b], w.dtype, f"{what} cuda cores seq {b}", v_scale)
    assert kvq.kvq_get_error() == (0, 0)


def _scaled(bits, dtype, factor, clip=None):
    x = bits_f64(bits, dtype) * factor
    if clip is not None:
        x = np.clip(x, -clip, clip)
    return W.to_bits(x.astype(np.float32), dtype)


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 128), (4, 4, 64)])
def test_decode_bf16_v_beyond_fp16_range(Hq, Hkv, D):
    """BF16 V of magnitude ~2^20 (absmax up to ~5e6, scales ~4e4): the
    product of a code and its scale is far beyond FP16's 65504.  One token
    also holds 8290304 (just below the saturation of the FP16 scale)."""
    w = W.custom(len(LENS), Hq, Hkv, D, "bf16", LENS, seed=201 + D)
    f = 2.0 ** 20
    seqs = []
    for b in range(w.num_seqs):
        k, v = w.seq_kv(b)
        v = _scaled(v, "bf16", f)
        if b == 3:
            v[5, 0, 7] = W.to_bits(np.array([8290304.0], np.float32), "bf16")[0]
            v[9, -1, 0] = W.to_bits(np.array([-8290304.0], np.float32), "bf16")[0]
        seqs.append((k, v))
    _decode_vs_oracle(w, seqs, w.q_all(), w.sm_scale, v_scale=f, what="bf16 V x2^20")


def test_decode_fp16_v_at_fp16_max():
    """FP16 V rows holding +-65504: the scale rounds up to 516 and 127 * 516
    = 65532 is above the largest FP16 number.  (Such a token's dequantized
    value itself exceeds FP16's range, so a context of that token alone has an
    infinite FP16 result; the extreme tokens go into contexts of 37 tokens
    and more, where the softmax spreads the weight.)"""
    w = W.custom(len(LENS), 8, 2, 128, "fp16", LENS, seed=211)
    f = 2.0 ** 13
    seqs = []
    r = np.random.default_rng(212)
    for b in range(w.num_seqs):
        k, v = w.seq_kv(b)
        v = _scaled(v, "fp16", f, clip=60000.0)
        L = len(v)
        if L >= 37:
            for t in r.choice(L, size=5, replace=False):
                v[t, r.integers(2), r.integers(128)] = 0x7BFF if t % 2 else 0xFBFF  # +-65504
        seqs.append((k, v))
    _decode_vs_oracle(w, seqs, w.q_all(), w.sm_scale, v_scale=f, what="fp16 V at 65504")


@pytest.mark.parametrize("qexp", [18, -20])
def test_decode_bf16_q_outside_fp16_normal_range(qexp):
    """BF16 queries times 2^18 (up to ~1e6) or 2^-20 (~1e-6, below FP16's
    normal range), with sm_scale times the inverse factor."""
    w = W.custom(len(LENS), 8, 2, 128, "bf16", LENS, seed=221 + qexp)
    seqs = [w.seq_kv(b) for b in range(w.num_seqs)]
    q = _scaled(w.q_all(), "bf16", 2.0 ** qexp)
    _decode_vs_oracle(w, seqs, q, w.sm_scale * 2.0 ** -qexp, what=f"bf16 q x2^{qexp}")


def test_decode_static_bf16_q_beyond_fp16_range():
    """The static-scale decode shares the query path: BF16 queries times 2^18."""
    w = W.custom(3, 8, 2, 128, "bf16", [16, 300, 1000], seed=231)
    case = Case(w)
    sk = sv = float(np.float32(5.0 / 127))
    kc, vc = case.int8[0], case.int8[1]
    seqs = [w.seq_kv(b) for b in range(w.num_seqs)]
    for b, (k, v) in enumerate(seqs):
        kvq.kvq_quantize_append_static(to_dev(k, "bf16"), to_dev(v, "bf16"),
                                       torch.from_numpy(w.slots(b, 0, len(k))).to("cuda"),
                                       kc, vc, sk, sv)
    f = 2.0 ** 18
    qb = _scaled(w.q_all(), "bf16", f)
    sm = w.sm_scale / f
    out = kvq.kvq_paged_decode_static(to_dev(qb, "bf16"), kc, vc, sk, sv, case.bt, case.cl,
                                      w.max_context_len, sm)
    ob = out_bits(out)
    for b, (k, v) in enumerate(seqs):
        kh = oracle.quantize_rows_static(k, "bf16", sk).astype(np.float64) * sk
        vh = oracle.quantize_rows_static(v, "bf16", sv).astype(np.float64) * sv
        qf = bits_f64(qb[b], "bf16")
        ref = np.stack([oracle.attend_one(qf[h], kh[:, h // 4], vh[:, h // 4], sm)
                        for h in range(8)])
        assert_attention_close(ob[b], ref, "bf16", f"static seq {b}")
    assert kvq.kvq_get_error() == (0, 0)


# ------------------------------------------------------------- prefill
def _queries(n, Hq, D, dtype, seed, factor=1.0):
    x = np.random.default_rng(seed).standard_normal((n, Hq, D)).astype(np.float32)
    return W.to_bits(x * np.float32(factor), dtype)


def _prefill_vs_oracle(w, seqs, chunks, qb, sm_scale, v_scale=1.0, what=""):
    case = Case(w)
    for b, (k, v) in enumerate(seqs):
        case._write(k, v, w.slots(b, 0, len(k)))
    qs = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32,
                      device="cuda")
    out = kvq.kvq_paged_prefill(to_dev(qb, w.dtype), *case.int8, case.bt, case.cl, qs,
                                w.max_context_len, max(chunks), sm_scale)
    ob = out_bits(out)
    start = 0
    for b, ((k, v), n) in enumerate(zip(seqs, chunks)):
        ref, _ = oracle.prefill_sequence(qb[start:start + n], k, v, w.dtype, sm_scale)
        for i in range(n):
            assert_attention_close(ob[start + i], ref[i], w.dtype, f"{what} seq {b} query {i}",
                                   v_scale)
        start += n
    assert kvq.kvq_get_error() == (0, 0)


@pytest.mark.parametrize("dtype,G", [("fp16", 1), ("bf16", 4), ("bf16", 8)])
def test_prefill_large_v_scales_under_growing_keys(dtype, G):
    """Keys growing along the sequence keep the softmax's probabilities up to
    2^8 between rescales; V of magnitude 2^14 (clipped to +-60000, whose
    dequantized values stay inside FP16, for both dtypes) has scales above
    256, so probability times scale passes 65504."""
    Hkv, D, L = 2, 128, 700
    w = W.custom(2, G * Hkv, Hkv, D, dtype, [L, 300], seed=241 + G)
    f = 2.0 ** 14
    seqs = []
    for b in range(2):
        k, v = w.seq_kv(b)
        kf = bits_f64(k, dtype) * (1.0 + 0.02 * np.arange(len(k)))[:, None, None]
        seqs.append((W.to_bits(kf.astype(np.float32), dtype),
                     _scaled(v, dtype, f, clip=60000.0)))
    chunks = [L, 77]
    qb = _queries(sum(chunks), G * Hkv, D, dtype, seed=242 + G)
    _prefill_vs_oracle(w, seqs, chunks, qb, w.sm_scale, v_scale=f, what=f"{dtype} V x2^14")


@pytest.mark.parametrize("qexp", [18, -20])
def test_prefill_bf16_q_outside_fp16_normal_range(qexp):
    Hkv, D = 2, 128
    w = W.custom(2, 8, Hkv, D, "bf16", [300, 129], seed=251 + qexp)
    seqs = [w.seq_kv(b) for b in range(2)]
    chunks = [300, 40]
    qb = _queries(sum(chunks), 8, D, "bf16", seed=252, factor=2.0 ** qexp)
    _prefill_vs_oracle(w, seqs, chunks, qb, w.sm_scale * 2.0 ** -qexp, what=f"q x2^{qexp}")
