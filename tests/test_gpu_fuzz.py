"""Seeded random shapes against the FP64 oracle.  Decode: for each case a random
batch, GQA ratio, head dim, dtype and ragged context lengths (including empty
and single-token sequences), appended (codes and scales read back through the
block tables, bit-exact), decoded by the tensor-core engine with the
launcher's balanced split, a random forced range length and no workspace, by
the CUDA-core engine, and by the 16-bit twin (against the oracle's native
attention); every (sequence, head) checked.  Chunked prefill: random shapes
and chunk lengths (empty, one query, the whole sequence, across CTA tiles),
every query row checked.  Static per-tensor scales: random shapes, codes
bit-exact, decode within tolerance.  The front trim and the dequantize-window
baseline: random shapes, bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import oracle
import workloads as W
from _harness import Case, assert_attention_close, out_bits, to_dev

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


def _chunk(rng, L):
    """A chunk length for a sequence of L tokens: empty, one query, the whole
    sequence, or a random length around the 64-token tile and the CTA edges."""
    pick = int(rng.integers(0, 5))
    if pick == 0 or L == 0:
        return 0 if pick == 0 else min(L, 1)
    if pick == 1:
        return 1
    if pick == 2:
        return L
    return int(rng.integers(1, L + 1))


@pytest.mark.parametrize("seed", range(40))
def test_prefill_random_shapes(seed):
    """Chunked prefill on seeded random shapes: every query row of every
    sequence against the oracle's causal attention over the dequantized
    tokens ("fix(cuda/kv): correct Int8 KV per-token scale ..." (mlxcel
    PR #717), "Server integration")."""
    rng = np.random.default_rng(3000 + seed)
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 5, 6, 7, 8]))
    D = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["fp16", "bf16"]))
    B = int(rng.integers(1, 5))
    lens = [int(x) for x in rng.choice([1, 2, 15, 16, 17, 63, 64, 65, 130, 300, 700], B)]
    chunks = [_chunk(rng, L) for L in lens]
    w = W.custom(B, G * Hkv, Hkv, D, dtype, lens, seed=4000 + seed)
    case = Case(w)
    case.write_prefix()
    x = rng.standard_normal((sum(chunks), w.num_q_heads, D)).astype(np.float32)
    qb = (x.astype(np.float16).view(np.uint16) if dtype == "fp16" else
          torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    qs = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32, device="cuda")
    q = torch.from_numpy(qb.view(np.int16)).to("cuda").view(
        torch.float16 if dtype == "fp16" else torch.bfloat16)
    out = kvq.kvq_paged_prefill(q, *case.int8, case.bt, case.cl, qs, w.max_context_len,
                                max(max(chunks), 1), w.sm_scale)
    ob = out_bits(out)
    what = f"Hkv={Hkv} G={G} D={D} {dtype} lens={lens} chunks={chunks}"
    start = 0
    for b, n in enumerate(chunks):
        if n:
            k, v = w.seq_kv(b)
            ref, _ = oracle.prefill_sequence(qb[start:start + n], k, v, dtype, w.sm_scale)
            for i in range(n):
                assert_attention_close(ob[start + i], ref[i], dtype, f"{what} seq {b} query {i}")
        start += n
    assert kvq.kvq_get_error() == (0, 0)


@pytest.mark.parametrize("seed", range(16))
def test_static_scale_random_shapes(seed):
    """The static per-tensor-scale variant ("fix: #552 int8 kv cache
    quantization cannot be enabled" (InfiniLM PR #553)) on seeded random
    shapes: codes bit-exact against the oracle's static quantizer, the decode
    (with and without a workspace) within tolerance of the oracle's attention
    over scale * code."""
    rng = np.random.default_rng(5000 + seed)
    Hkv, G, D, dtype, lens = _shape(rng)
    w = W.custom(len(lens), G * Hkv, Hkv, D, dtype, lens, seed=6000 + seed)
    case = Case(w)
    # calibrated scales (max |x| / 127 over the workload), or a shared or unit one
    mk = mv = 0.0
    for b in range(w.num_seqs):
        k, v = w.seq_kv(b)
        if len(k):
            mk = max(mk, float(np.abs(oracle.bits_to_double(k, dtype)).max()))
            mv = max(mv, float(np.abs(oracle.bits_to_double(v, dtype)).max()))
    sk, sv = float(np.float32(max(mk, 1e-3) / 127)), float(np.float32(max(mv, 1e-3) / 127))
    mode = int(rng.integers(0, 3))
    if mode == 1:
        sk = sv = max(sk, sv)
    elif mode == 2:
        sk = sv = 1.0
    kc, vc = case.int8[0], case.int8[1]
    for b in range(w.num_seqs):
        k, v = w.seq_kv(b)
        if len(k):
            s = torch.from_numpy(w.slots(b, 0, len(k))).to("cuda")
            kvq.kvq_quantize_append_static(to_dev(k, dtype), to_dev(v, dtype), s, kc, vc, sk, sv)
    none = torch.empty(0, dtype=torch.uint8, device="cuda")
    outs = {"balanced": kvq.kvq_paged_decode_static(case.q, kc, vc, sk, sv, case.bt, case.cl,
                                                    w.max_context_len, w.sm_scale),
            "no workspace": kvq.kvq_paged_decode_static(case.q, kc, vc, sk, sv, case.bt, case.cl,
                                                        w.max_context_len, w.sm_scale,
                                                        workspace=none)}
    what = f"Hkv={Hkv} G={G} D={D} {dtype} lens={lens} scales=({sk}, {sv})"
    for b in range(w.num_seqs):
        k, v = w.seq_kv(b)
        ck, cv, _, _ = case.gather_seq(b)
        wk = oracle.quantize_rows_static(k, dtype, sk)
        wv = oracle.quantize_rows_static(v, dtype, sv)
        assert np.array_equal(ck, wk), f"{what} seq {b}: K codes"
        assert np.array_equal(cv, wv), f"{what} seq {b}: V codes"
        if len(k) == 0:
            ref = np.zeros((w.num_q_heads, D))
        else:
            kh, vh = wk.astype(np.float64) * sk, wv.astype(np.float64) * sv
            qf = oracle.bits_to_double(w.seq_q(b), dtype)
            ref = np.stack([oracle.attend_one(qf[h], kh[:, h // G], vh[:, h // G], w.sm_scale)
                            for h in range(w.num_q_heads)])
        for name, out in outs.items():
            assert_attention_close(out_bits(out)[b], ref, dtype, f"{what} {name} seq {b}")
    assert kvq.kvq_get_error() == (0, 0)


def _cache_rows(case, b, L):
    """(K codes, V codes, K scale bits, V scale bits) of sequence b's first L
    tokens read back through its block table."""
    t = torch.arange(L, device="cuda")
    blk = case.bt[b, t // 16].long()
    off = t % 16
    kc, vc, ks, vs = case.int8
    return [kc[blk, :, off].cpu().numpy(), vc[blk, :, off].cpu().numpy(),
            ks[blk, :, off].cpu().numpy(), vs[blk, :, off].cpu().numpy()]


@pytest.mark.parametrize("seed", range(16))
def test_trim_random_shapes(seed):
    """Front trim keeping the sink ("fix(cuda/kv): correct Int8 KV per-token
    scale ..." (mlxcel PR #717), follow-up commit) on seeded random shapes,
    sink lengths and trims (zero, within, past the length): the rows and
    scales left equal the oracle's trim bit for bit, context_lens follows."""
    rng = np.random.default_rng(7000 + seed)
    Hkv, G, D, dtype, lens = _shape(rng)
    keep = int(rng.choice([0, 1, 4, 16, 33]))
    trims = [int(rng.choice([0, 1, 15, 16, 17, max(L - keep, 0), L + 5]))
             if rng.random() < 0.5 else int(rng.integers(0, L + 2)) for L in lens]
    w = W.custom(len(lens), G * Hkv, Hkv, D, dtype, lens, seed=8000 + seed)
    case = Case(w)
    case.write_prefix()
    before = [_cache_rows(case, b, L) for b, L in enumerate(lens)]
    tr = torch.tensor(trims, dtype=torch.int32, device="cuda")
    kvq.kvq_trim_front_keep_sink(*case.int8, case.bt, case.cl, tr, keep)
    new_lens = case.cl.cpu().numpy()
    what = f"Hkv={Hkv} D={D} lens={lens} keep={keep} trims={trims}"
    for b, L in enumerate(lens):
        n = max(0, min(trims[b], L - min(keep, L)))
        assert new_lens[b] == L - n, f"{what} seq {b}: length"
        after = _cache_rows(case, b, L - n)
        for x, y in zip(before[b], after):
            assert np.array_equal(oracle.trim_keep_sink(x, keep, trims[b]), y), f"{what} seq {b}"
    assert kvq.kvq_get_error() == (0, 0)


@pytest.mark.parametrize("seed", range(16))
def test_dequantize_window_random_shapes(seed):
    """The dequantize-window baseline ("fix(cuda/kv): correct Int8 KV per-token
    scale ..." (mlxcel PR #717), "The Int8 bug and fix") on seeded random
    shapes: every valid token's 16-bit value equals the oracle's code * scale
    rounded once to the dtype."""
    rng = np.random.default_rng(9000 + seed)
    Hkv, G, D, dtype, lens = _shape(rng)
    w = W.custom(len(lens), G * Hkv, Hkv, D, dtype, lens, seed=9500 + seed)
    case = Case(w)
    case.write_prefix()
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    kw, vw = kvq.kvq_dequantize_window(*case.int8, case.bt, case.cl, w.max_context_len, tdt)
    torch.cuda.synchronize()
    for b, L in enumerate(lens):
        t = torch.arange(L, device="cuda")
        blk = case.bt[b, t // 16].long()
        off = t % 16
        got = [x[blk, :, off].cpu().view(torch.int16).numpy().view(np.uint16) for x in (kw, vw)]
        k, v = w.seq_kv(b)
        for x, g, nm in ((k, got[0], "K"), (v, got[1], "V")):
            q, s = oracle.quantize_rows(x, dtype)
            assert np.array_equal(g, oracle.dequantize_rows(q, s, dtype)), (
                f"Hkv={Hkv} D={D} {dtype} lens={lens} seq {b} {nm}")
    assert kvq.kvq_get_error() == (0, 0)
