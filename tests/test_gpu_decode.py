"""Paged decode on the GPU against the FP64 oracle: every workload (full size,
through the launcher the benchmark uses), every launcher variant (forced
partition sizes), ragged and degenerate contexts, GQA ratios, both head dims
and dtypes, the 16-bit twin, and the device/host error paths."""
import ctypes

import numpy as np
import pytest
import torch

import int8_quantized_paged_tokenwise_gb300 as kvq
import oracle
import workloads as W
from _harness import Case, assert_attention_close, out_bits

pytestmark = pytest.mark.gpu


def _oracle_seq(w, b, quantized=True, heads=None):
    k, v = w.seq_kv(b)
    out, _ = oracle.decode_sequence(w.seq_q(b), k, v, w.dtype, w.sm_scale,
                                    quantized=quantized, heads=heads)
    return out


def _check_all(case, out, quantized=True, what=""):
    w = case.w
    ob = out_bits(out)
    errs = []
    for b in range(w.num_seqs):
        errs.append(assert_attention_close(ob[b], _oracle_seq(w, b, quantized), w.dtype,
                                           f"{what} seq {b}"))
    return max(errs) if errs else 0.0


def _check_sampled(case, out, n_pairs, seed=0, quantized=True, what="", seqs=None):
    w = case.w
    ob = out_bits(out)
    r = np.random.default_rng(seed)
    bs = seqs if seqs is not None else r.choice(w.num_seqs, size=min(n_pairs, w.num_seqs),
                                                replace=False)
    for b in bs:
        heads = sorted(r.choice(w.num_q_heads, size=min(4, w.num_q_heads), replace=False))
        ref = _oracle_seq(w, int(b), quantized, heads=heads)
        assert_attention_close(ob[b, heads], ref, w.dtype, f"{what} seq {b} heads {heads}")


# ----------------------------------------------------------------- workloads
def test_decode_tiny_all_variants():
    case = Case(W.make("tiny"), kv16=True)
    case.write_prefix()
    case.write_step()
    for P in (0, 4, 8, 1024):
        _check_all(case, case.decode(P), what=f"tiny P={P}")
        _check_all(case, case.decode(P, kv16=True), quantized=False, what=f"tiny kv16 P={P}")
    assert kvq.kvq_get_error() == (0, 0)


def test_decode_canonical_full():
    """Every (sequence, head) of the canonical GQA workload after one step."""
    case = Case(W.make("canonical"), kv16=True)
    case.write_prefix()
    case.write_step()
    _check_all(case, case.decode(), what="canonical")
    _check_all(case, case.decode(kv16=True), quantized=False, what="canonical kv16")
    for P in (4, 16, 64):
        _check_sampled(case, case.decode(P), 6, seed=P, what=f"canonical P={P}")
    assert kvq.kvq_get_error() == (0, 0)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["long", "mha", "serving"])
def test_decode_full_workload_sampled(name):
    """Full-size workloads through the launcher, sampled (sequence, head) pairs
    against the oracle; the 16-bit twin likewise."""
    w = W.make(name)
    case = Case(w, kv16=True)
    case.write_prefix()
    case.write_step()
    out = case.decode()
    _check_sampled(case, out, 6, seed=1, what=name)
    _check_sampled(case, case.decode(kv16=True), 3, seed=2, quantized=False, what=name + " kv16")
    if name == "serving":
        # the fragmented split-K extremes: the longest sequences (many ranges
        # each) and the shortest (a piece of a single page)
        order = np.argsort(w.context_lens, kind="stable")
        _check_sampled(case, out, 0, seed=5, what="serving extremes",
                       seqs=[int(b) for b in (*order[:3], *order[-3:])])
    assert bool(torch.isfinite(out.float()).all())
    assert kvq.kvq_get_error() == (0, 0)


# ------------------------------------------------------------ ragged / edges
RAGGED = [0, 1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 250, 513, 1000, 2049, 4100]


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(4, 2, 64, "fp16"), (32, 8, 128, "bf16"),
                                            (8, 8, 128, "fp16"), (16, 2, 64, "bf16"),
                                            (12, 4, 128, "fp16"), (5, 1, 64, "bf16")])
def test_decode_ragged_contexts_every_partition_size(Hq, Hkv, D, dtype):
    w = W.custom(len(RAGGED), Hq, Hkv, D, dtype, RAGGED, seed=Hq * 7 + D)
    case = Case(w, kv16=True)
    case.write_prefix()
    for P in (0, 4, 8, 12, 32, 64, 300):
        P = P if P % 4 == 0 else P - P % 4
        out = case.decode(P)
        _check_all(case, out, what=f"ragged P={P}")
        # empty context -> exact zeros
        assert bool((out[0] == 0).all())
    _check_all(case, case.decode(8, kv16=True), quantized=False, what="ragged kv16")
    assert kvq.kvq_get_error() == (0, 0)


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(4, 4, 128, "fp16"), (8, 4, 64, "bf16"),
                                            (32, 8, 128, "bf16"), (16, 2, 128, "bf16"),
                                            (12, 4, 64, "fp16")])
def test_decode_cuda_cores_matches_oracle(Hq, Hkv, D, dtype):
    """The CUDA-core engine (the tensor cores' A/B counterpart) over ragged
    contexts, G in {1, 2, 3, 4, 8}: split-K with the recommended workspace and
    one range per sequence without one."""
    w = W.custom(len(RAGGED), Hq, Hkv, D, dtype, RAGGED, seed=Hq * 11 + D + 5)
    case = Case(w)
    case.write_prefix()
    out = kvq.kvq_paged_decode_cuda_cores(case.q, *case.int8, case.bt, case.cl,
                                          w.max_context_len, w.sm_scale)
    _check_all(case, out, what="cuda cores")
    assert bool((out[0] == 0).all())
    none = torch.empty(0, dtype=torch.uint8, device="cuda")
    out = kvq.kvq_paged_decode_cuda_cores(case.q, *case.int8, case.bt, case.cl,
                                          w.max_context_len, w.sm_scale, workspace=none)
    _check_all(case, out, what="cuda cores, no workspace")
    assert kvq.kvq_get_error() == (0, 0)


def test_decode_single_token_returns_v():
    w = W.custom(3, 8, 2, 128, "bf16", [1, 1, 1], seed=3)
    case = Case(w)
    case.write_prefix()
    ob = out_bits(case.decode())
    for b in range(3):
        k, v = w.seq_kv(b)
        qv, sv = oracle.quantize_rows(v, "bf16")
        for h in range(8):
            vh = qv[0, h // 4].astype(np.float64) * oracle.fp16_to_double(int(sv[0, h // 4]))
            assert_attention_close(ob[b, h][None], vh[None], "bf16", "single token")


def test_decode_equal_keys_mean_of_v():
    w = W.custom(2, 4, 2, 64, "fp16", [37, 200], seed=4)
    case = Case(w)
    # overwrite: every key of a sequence identical -> uniform softmax
    for b in range(2):
        k, v = w.seq_kv(b)
        k[:] = k[0]
        case._write(k, v, w.slots(b, 0, len(k)))
    ob = out_bits(case.decode(4))
    for b in range(2):
        k, v = w.seq_kv(b)
        qv, sv = oracle.quantize_rows(v, "fp16")
        vhat = qv.astype(np.float64) * oracle.bits_to_double(sv, "fp16")[..., None]
        mean = vhat.mean(axis=0)
        for h in range(4):
            assert_attention_close(ob[b, h][None], mean[h // 2][None], "fp16", "equal keys")


def test_decode_zero_tokens_use_unit_scale_and_contribute_zero_values():
    w = W.custom(2, 4, 4, 128, "fp16", [100, 64], seed=9, zero_token_frac=0.1)
    case = Case(w)
    case.write_prefix()
    _check_all(case, case.decode(), what="zero tokens")
    k, v = w.seq_kv(0)
    zero_rows = np.where(~k.any(axis=(1, 2)))[0]
    assert len(zero_rows) == 10
    gk, gv, gks, gvs = case.gather_seq(0)
    assert np.all(gks[zero_rows] == 0x3C00) and np.all(gk[zero_rows] == 0)


def test_decode_large_scores_stable():
    """Large-magnitude q and K (outlier channels) exercise the running max."""
    w = W.custom(4, 8, 2, 128, "bf16", [3000, 17, 700, 1], seed=10, q_std=8.0,
                 outlier_channels=4, outlier_gain=30.0)
    case = Case(w)
    case.write_prefix()
    for P in (0, 4, 16):
        _check_all(case, case.decode(P), what=f"large scores P={P}")


def test_decode_repeated_calls_deterministic():
    w = W.make("canonical")
    case = Case(w)
    case.write_prefix()
    a = case.decode().clone()
    b = case.decode().clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# -------------------------------------------------------------- error paths
def test_decode_bad_block_id_sets_error_bit():
    w = W.custom(2, 4, 2, 64, "fp16", [40, 40], seed=6)
    case = Case(w)
    case.write_prefix()
    case.bt[1, 1] = case.nb + 5                      # out of range
    out = case.decode(4)
    st, flags = kvq.kvq_get_error()
    assert st == 5 and flags & kvq.DEVERR_BLOCK
    ob = out_bits(out)
    assert_attention_close(ob[0], _oracle_seq(w, 0), "fp16", "healthy seq")
    case.bt[1, 1] = -3
    case.decode()
    st, flags = kvq.kvq_get_error()
    assert flags & kvq.DEVERR_BLOCK


def test_decode_context_beyond_table_sets_error_bit():
    w = W.custom(2, 4, 2, 64, "fp16", [40, 40], seed=7)
    case = Case(w)
    case.write_prefix()
    case.cl[1] = case.bt.shape[1] * 16 + 1
    case.decode()
    st, flags = kvq.kvq_get_error()
    assert st == 5 and flags & kvq.DEVERR_CONTEXT
    assert kvq.kvq_get_error() == (0, 0)


def test_decode_context_beyond_host_bound_is_clamped():
    """A context above the host's max_context_len (but inside the table) is
    flagged and clamped, so split partials never outgrow the workspace."""
    w = W.custom(2, 4, 2, 64, "fp16", [100, 40], seed=12)
    case = Case(w)
    case.write_prefix()
    out = kvq.kvq_paged_decode(case.q, *case.int8, case.bt, case.cl, 60, w.sm_scale,
                               partition_pages=4)
    st, flags = kvq.kvq_get_error()
    assert st == 5 and flags & kvq.DEVERR_CONTEXT
    assert_attention_close(out_bits(out)[1], _oracle_seq(w, 1), "fp16", "in-bound seq")


def test_decode_host_validation():
    w = W.custom(2, 4, 2, 64, "fp16", [100, 40], seed=8)
    case = Case(w)
    L = kvq.load()
    kc, vc, ks, vs = case.int8
    P = ctypes.c_void_p
    out = torch.empty_like(case.q)

    def call(**kw):
        a = dict(q=P(case.q.data_ptr()), dtype=0, B=2, Hq=4, Hkv=2, D=64, kc=P(kc.data_ptr()),
                 vc=P(vc.data_ptr()), ks=P(ks.data_ptr()), vs=P(vs.data_ptr()), nb=case.nb, bs=16,
                 bt=P(case.bt.data_ptr()), mb=case.bt.shape[1], cl=P(case.cl.data_ptr()),
                 mc=100, scale=0.125, out=P(out.data_ptr()), ws=None, wsb=0)
        a.update(kw)
        return L.kvq_paged_decode(*a.values(), None)

    assert call() == 0
    assert call(Hq=5) == 1                            # Hq % Hkv
    assert call(Hq=18) == 2                           # group 9 > 8
    assert call(D=96) == 2
    assert call(bs=8) == 2
    assert call(kc=None) == 1
    assert call(ks=None) == 1
    assert call(q=P(case.q.data_ptr() + 2)) == 1      # misaligned
    assert call(mc=case.bt.shape[1] * 16 + 1) == 1    # host bound beyond the table
    assert call(scale=float("nan")) == 1
    assert call(B=0) == 0                             # empty batch: no-op
    # a split that needs workspace, given none
    assert L.kvq_paged_decode_split(P(case.q.data_ptr()), 0, 2, 4, 2, 64, P(kc.data_ptr()),
                                    P(vc.data_ptr()), P(ks.data_ptr()), P(vs.data_ptr()), case.nb,
                                    16, P(case.bt.data_ptr()), case.bt.shape[1],
                                    P(case.cl.data_ptr()), 100, 0.125, P(out.data_ptr()), None, 0,
                                    4, None) == 4
    assert L.kvq_paged_decode_split(P(case.q.data_ptr()), 0, 2, 4, 2, 64, P(kc.data_ptr()),
                                    P(vc.data_ptr()), P(ks.data_ptr()), P(vs.data_ptr()), case.nb,
                                    16, P(case.bt.data_ptr()), case.bt.shape[1],
                                    P(case.cl.data_ptr()), 100, 0.125, P(out.data_ptr()), None, 0,
                                    0, None) == 1     # no partition size
    torch.cuda.synchronize()
    assert kvq.kvq_get_error() == (0, 0)


def test_decode_on_side_stream_and_graph_capture():
    """The calls are stream-ordered, allocate nothing and can be captured in a
    CUDA graph (workspace preallocated)."""
    w = W.make("canonical")
    case = Case(w)
    case.write_prefix()
    ref = case.decode().clone()
    ws = torch.empty(max(1, kvq.kvq_decode_workspace_bytes(w.num_seqs, w.num_q_heads,
                                                           w.num_kv_heads, w.head_dim,
                                                           w.max_context_len)),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(case.q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kvq.kvq_paged_decode(case.q, *case.int8, case.bt, case.cl, w.max_context_len,
                             w.sm_scale, out=out, workspace=ws)
    s.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        kvq.kvq_paged_decode(case.q, *case.int8, case.bt, case.cl, w.max_context_len,
                             w.sm_scale, out=out, workspace=ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_decode_without_workspace_and_with_a_small_one():
    """An empty workspace runs one warp per (sequence, KV head) with no split;
    a workspace for only a few work ranges lowers the warp count (long
    ranges, many pieces per range).  Both match the oracle."""
    w = W.custom(len(RAGGED), 16, 4, 128, "bf16", RAGGED, seed=31)
    case = Case(w)
    case.write_prefix()
    none = torch.empty(0, dtype=torch.uint8, device="cuda")
    out = kvq.kvq_paged_decode(case.q, *case.int8, case.bt, case.cl, w.max_context_len,
                               w.sm_scale, workspace=none)
    _check_all(case, out, what="no workspace")
    assert bool((out[0] == 0).all())
    for ranges_pages in (w.max_context_len, 64):
        # bytes for ceil(tiles / ranges_pages) ranges: a handful of ranges
        nbytes = kvq.kvq_decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                                w.head_dim, w.max_context_len, ranges_pages)
        small = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        out = kvq.kvq_paged_decode(case.q, *case.int8, case.bt, case.cl, w.max_context_len,
                                   w.sm_scale, workspace=small)
        _check_all(case, out, what=f"small workspace ({nbytes} B)")
    assert kvq.kvq_get_error() == (0, 0)


@pytest.mark.parametrize("Hq,Hkv,D,dtype", [(8, 2, 128, "bf16"), (4, 4, 64, "fp16")])
def test_decode_short_contexts_take_the_unsplit_path(Hq, Hkv, D, dtype):
    """Contexts of at most four pages (64 tokens) are never split: with the
    recommended workspace (0 bytes for such calls) and with a large one the
    output is the no-workspace output bit for bit, and every sequence matches
    the oracle; a 65-token bound goes back to the split path."""
    lens = [0, 1, 15, 16, 17, 33, 48, 63, 64] * 3
    w = W.custom(len(lens), Hq, Hkv, D, dtype, lens, seed=91 + Hq)
    assert w.max_context_len <= 64
    case = Case(w)
    case.write_prefix()
    assert kvq.kvq_decode_workspace_bytes(w.num_seqs, Hq, Hkv, D, w.max_context_len) == 0
    none = torch.empty(0, dtype=torch.uint8, device="cuda")
    ref = kvq.kvq_paged_decode(case.q, *case.int8, case.bt, case.cl, w.max_context_len,
                               w.sm_scale, workspace=none)
    _check_all(case, ref, what="short contexts")
    big = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    out = kvq.kvq_paged_decode(case.q, *case.int8, case.bt, case.cl, w.max_context_len,
                               w.sm_scale, workspace=big)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert kvq.kvq_decode_workspace_bytes(w.num_seqs, Hq, Hkv, D, 65) > 0
    assert kvq.kvq_get_error() == (0, 0)
