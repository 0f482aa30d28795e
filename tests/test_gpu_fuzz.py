"""Seeded random shapes against the FP64 oracle: for each case a random
batch, GQA ratio, head dim, dtype and ragged context lengths (including empty
and single-token sequences), appended (codes and scales read back through the
block tables, bit-exact), decoded by the tensor-core engine with the
launcher's balanced split, a random forced range length and no workspace, by
the CUDA-core engine, and by the 16-bit twin (against the oracle's native
attention); every (sequence, head) checked."""
import numpy as np
import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import oracle
import workloads as W
from _harness import Case, assert_attention_close, out_bits

pytestmark = pytest.mark.gpu


def _shape(rng):
    Hkv = int(rng.choice([1, 2, 3, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8]))
    D = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["fp16", "bf16"]))
    B = int(rng.integers(1, 9))
    lens = [int(x) for x in rng.choice([0, 1, 2, 15, 16, 17, 31, 64, 65, 100, 257, 700, 1500], B)]
    return Hkv, G, D, dtype, lens


@pytest.mark.parametrize("seed", range(40))
def test_decode_random_shapes(seed):
    rng = np.random.default_rng(1000 + seed)
    Hkv, G, D, dtype, lens = _shape(rng)
    w = W.custom(len(lens), G * Hkv, Hkv, D, dtype, lens, seed=2000 + seed)
    case = Case(w, kv16=True)
    case.write_prefix()
    refs = [oracle.decode_sequence(w.seq_q(b), *w.seq_kv(b), w.dtype, w.sm_scale)[0]
            for b in range(w.num_seqs)]
    refs16 = [oracle.decode_sequence(w.seq_q(b), *w.seq_kv(b), w.dtype, w.sm_scale,
                                     quantized=False)[0] for b in range(w.num_seqs)]
    R = int(rng.integers(1, 40))
    none = torch.empty(0, dtype=torch.uint8, device="cuda")
    outs = {
        "balanced": case.decode(),
        f"forced R={R}": case.decode(partition_pages=R),
        "no workspace": kvq.kvq_paged_decode(case.q, *case.int8, case.bt, case.cl,
                                             w.max_context_len, w.sm_scale, workspace=none),
        "cuda cores": kvq.kvq_paged_decode_cuda_cores(case.q, *case.int8, case.bt, case.cl,
                                                      w.max_context_len, w.sm_scale),
    }
    what = f"Hkv={Hkv} G={G} D={D} {dtype} lens={lens}"
    for b in range(w.num_seqs):
        k, v = w.seq_kv(b)
        gk, gv, gks, gvs = case.gather_seq(b)
        for x, gc, gs, nm in ((k, gk, gks, "K"), (v, gv, gvs, "V")):
            qc, qs = oracle.quantize_rows(x, w.dtype)
            assert np.array_equal(gs, qs), f"{what} seq {b}: {nm} scales differ"
            assert np.array_equal(gc, qc), f"{what} seq {b}: {nm} codes differ"
    for name, out in outs.items():
        ob = out_bits(out)
        for b in range(w.num_seqs):
            assert_attention_close(ob[b], refs[b], w.dtype, f"{what} {name} seq {b}")
    # the twin's P V runs on 16-bit operands of the cache's type: with BF16 the
    # softmax weights carry 8 significant bits, a relative error up to 2^-9 on
    # each weight and so up to 2^-9 max|v| on the output (visible with a few
    # tokens, where no averaging hides it); FP16 weights stay inside the bound
    ob = out_bits(case.decode(kv16=True))
    for b in range(w.num_seqs):
        extra = 0.0
        if dtype == "bf16" and lens[b] > 0:
            vb = w.seq_kv(b)[1]
            vmax = float(np.abs((vb.astype(np.uint32) << 16).view(np.float32)).max())
            extra = 2.0 ** -9 * vmax
        assert_attention_close(ob[b], refs16[b], w.dtype, f"{what} 16-bit twin seq {b}",
                               atol_extra=extra)
    assert kvq.kvq_get_error() == (0, 0)
