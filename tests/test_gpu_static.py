"""The static-scale variant through the C ABI: one binary32 scale per tensor
("fix: #552 int8 kv cache quantization cannot be enabled" (InfiniLM PR #553);
"Add calibrated INT8 KV cache to PyTorch backend" (TensorRT-LLM PR #18953)).

* Quantize-on-write is bit-exact against the oracle's static quantizer on
  every token of ragged workloads (calibrated scales, the default 1.0, and a
  scale shared by K and V).
* The decode over that cache matches the oracle's attention over
  scale * code within the attention tolerance.
* Host validation of the scales.
"""
import numpy as np
import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import oracle
import workloads as W
from _harness import BS, Case, assert_attention_close, out_bits, to_dev

pytestmark = pytest.mark.gpu

RAGGED = [0, 1, 15, 16, 17, 100, 513, 2049]


def _calibrate(w):
    """Per-tensor scales max|x| / 127 over every token of the workload (binary32)."""
    mk = mv = 0.0
    for b in range(w.num_seqs):
        k, v = w.seq_kv(b)
        if len(k):
            mk = max(mk, float(np.abs(oracle.bits_to_double(k, w.dtype)).max()))
            mv = max(mv, float(np.abs(oracle.bits_to_double(v, w.dtype)).max()))
    return float(np.float32(mk / 127)), float(np.float32(mv / 127))


def _write_static(case, sk, sv):
    w = case.w
    kc, vc = case.int8[0], case.int8[1]
    for b in range(w.num_seqs):
        k, v = w.seq_kv(b)
        n = len(k)
        if n == 0:
            continue
        s = torch.from_numpy(w.slots(b, 0, n)).to("cuda")
        kvq.kvq_quantize_append_static(to_dev(k, w.dtype), to_dev(v, w.dtype), s, kc, vc, sk, sv)


@pytest.mark.parametrize("Hq,Hkv,D,dtype,mode", [(8, 2, 128, "bf16", "calibrated"),
                                                 (4, 4, 64, "fp16", "calibrated"),
                                                 (12, 4, 128, "fp16", "shared"),
                                                 (8, 2, 64, "bf16", "unit")])
def test_static_quantize_bit_exact_and_decode(Hq, Hkv, D, dtype, mode):
    w = W.custom(len(RAGGED), Hq, Hkv, D, dtype, RAGGED, seed=61 + D + Hq)
    case = Case(w)
    sk, sv = _calibrate(w)
    if mode == "shared":
        sk = sv = max(sk, sv)
    elif mode == "unit":
        sk = sv = 1.0
    _write_static(case, sk, sv)
    out = kvq.kvq_paged_decode_static(case.q, case.int8[0], case.int8[1], sk, sv, case.bt,
                                      case.cl, w.max_context_len, w.sm_scale)
    ob = out_bits(out)
    for b in range(w.num_seqs):
        L = int(w.context_lens[b])
        k, v = w.seq_kv(b)
        ck, cv, _, _ = case.gather_seq(b)
        wk = oracle.quantize_rows_static(k, dtype, sk)
        wv = oracle.quantize_rows_static(v, dtype, sv)
        assert np.array_equal(ck, wk[:L]), f"seq {b} K codes"
        assert np.array_equal(cv, wv[:L]), f"seq {b} V codes"
        kh = wk.astype(np.float64) * sk
        vh = wv.astype(np.float64) * sv
        qf = oracle.bits_to_double(w.seq_q(b), dtype)
        G = Hq // Hkv
        ref = np.stack([oracle.attend_one(qf[h], kh[:, h // G], vh[:, h // G], w.sm_scale)
                        for h in range(Hq)])
        assert_attention_close(ob[b], ref, dtype, f"static decode seq {b}")
    assert kvq.kvq_get_error() == (0, 0)


def test_static_scale_validation():
    w = W.custom(2, 4, 2, 64, "fp16", [20, 20], seed=63)
    case = Case(w)
    k, v = w.seq_kv(0)
    s = torch.from_numpy(w.slots(0, 0, len(k))).to("cuda")
    for bad in (0.0, -1.0, float("nan"), float("inf"), 1e-45):
        with pytest.raises(kvq.KvqError):
            kvq.kvq_quantize_append_static(to_dev(k, "fp16"), to_dev(v, "fp16"), s,
                                           case.int8[0], case.int8[1], bad, 1.0)
        if bad == 1e-45:          # a subnormal scale is a valid decode scale (no reciprocal)
            continue
        with pytest.raises(kvq.KvqError):
            kvq.kvq_paged_decode_static(case.q, case.int8[0], case.int8[1], 1.0, bad, case.bt,
                                        case.cl, w.max_context_len, w.sm_scale)
    torch.cuda.synchronize()
    assert kvq.kvq_get_error() == (0, 0)
