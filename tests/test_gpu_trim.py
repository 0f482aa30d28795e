"""Front trim keeping the attention sink ("fix(cuda/kv): correct Int8 KV
per-token scale ..." (mlxcel PR #717), follow-up commit, "The fix") through
the C ABI: payload and scale rows move in lockstep, bit-exact against the
oracle's trim of the sequence's rows; context_lens is updated; the decode
over the trimmed cache matches the oracle's attention over the trimmed
tokens; a static-scale cache (no scale planes) trims its codes."""
import numpy as np
import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import oracle
import workloads as W
from _harness import BS, Case, assert_attention_close, out_bits, to_dev

pytestmark = pytest.mark.gpu

LENS = [0, 3, 17, 40, 100, 513, 1000, 2049]
TRIMS = [5, 2, 20, 1, 37, 300, 0, 1500]


def _rows(case, b, L, planes=True):
    t = torch.arange(L, device="cuda")
    blk = case.bt[b, t // BS].long()
    off = t % BS
    kc, vc, ks, vs = case.int8
    out = [kc[blk, :, off].cpu().numpy(), vc[blk, :, off].cpu().numpy()]
    if planes:
        out += [ks[blk, :, off].cpu().numpy(), vs[blk, :, off].cpu().numpy()]
    return out


@pytest.mark.parametrize("keep", [4, 0, 33])
def test_trim_keep_sink_moves_rows_and_scales(keep):
    w = W.custom(len(LENS), 8, 2, 128, "bf16", LENS, seed=71 + keep)
    case = Case(w)
    case.write_prefix()
    before = [_rows(case, b, int(L)) for b, L in enumerate(LENS)]
    trim = torch.tensor(TRIMS, dtype=torch.int32, device="cuda")
    kvq.kvq_trim_front_keep_sink(*case.int8, case.bt, case.cl, trim, keep)
    new_lens = case.cl.cpu().numpy()
    out = kvq.kvq_paged_decode(case.q, *case.int8, case.bt, case.cl, w.max_context_len, w.sm_scale)
    ob = out_bits(out)
    for b, L in enumerate(LENS):
        kb = min(keep, L)
        n = max(0, min(TRIMS[b], L - kb))
        assert new_lens[b] == L - n, f"seq {b} length"
        after = _rows(case, b, L - n)
        for x, y in zip(before[b], after):
            assert np.array_equal(oracle.trim_keep_sink(x, keep, TRIMS[b]), y), f"seq {b}"
        k, v = w.seq_kv(b)
        ref, _ = oracle.decode_sequence(w.seq_q(b), oracle.trim_keep_sink(k, keep, TRIMS[b]),
                                        oracle.trim_keep_sink(v, keep, TRIMS[b]), "bf16",
                                        w.sm_scale)
        assert_attention_close(ob[b], ref, "bf16", f"decode after trim seq {b}")
    assert kvq.kvq_get_error() == (0, 0)


def test_trim_static_cache_codes_only():
    w = W.custom(3, 4, 4, 64, "fp16", [300, 64, 9], seed=77)
    case = Case(w)
    kc, vc = case.int8[0], case.int8[1]
    for b in range(3):
        k, v = w.seq_kv(b)
        s = torch.from_numpy(w.slots(b, 0, len(k))).to("cuda")
        kvq.kvq_quantize_append_static(to_dev(k, "fp16"), to_dev(v, "fp16"), s, kc, vc, 0.02, 0.03)
    before = [_rows(case, b, int(L), planes=False) for b, L in enumerate(w.context_lens)]
    trim = torch.tensor([250, 64, 3], dtype=torch.int32, device="cuda")
    kvq.kvq_trim_front_keep_sink(kc, vc, None, None, case.bt, case.cl, trim, 4)
    lens = case.cl.cpu().numpy()
    assert lens.tolist() == [50, 4, 6]
    for b in range(3):
        after = _rows(case, b, int(lens[b]), planes=False)
        for x, y in zip(before[b], after):
            assert np.array_equal(oracle.trim_keep_sink(x, 4, int(trim[b])), y)
    assert kvq.kvq_get_error() == (0, 0)
