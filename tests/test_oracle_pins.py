"""Pins of the FP64 oracle to facts outside itself (CPU only).

Each check below is chosen so that a plausible slip in the oracle (a dropped
term, a wrong sign or index, a transposed operand, the wrong rounding
direction) fails at least one of them:

* 16-bit decoders/encoders against numpy's float16 and torch's bfloat16
  (independent library routines), exhaustively or on exact halfway points;
* the quantizer against the facts the pages state (error bound, no -128, exact
  zero, all-zero token -> scale 1.0, largest coordinate -> +-127), against
  exact rational arithmetic (``fractions``) and brute force over fp16 bands;
* the page-byte formula against the figure printed on the page;
* attention against torch's float64 scaled_dot_product_attention (a library
  routine, GQA by consecutive grouping), closed forms (single token, equal
  keys) and the partitioned log-sum-exp formulation.
"""
from fractions import Fraction
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _facts():
    out = {}
    with open(os.path.join(GOLDEN, "quantizer_facts.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, val, _src = [s.strip() for s in line.split("|")]
            out[name] = float(int(val, 16)) if val.startswith("0x") else float(val)
    return out


FACTS = _facts()


# ------------------------------------------------------------ 16-bit formats
def test_fp16_decode_exhaustive_vs_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(ref[fin]))
    assert np.all(np.isinf(got[np.isinf(ref)])) and np.all(np.isnan(got[np.isnan(ref)]))


def test_bf16_decode_exhaustive_vs_torch():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = oracle.bits_to_double(bits, "bf16")
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.all(np.isnan(got[np.isnan(ref)]))


def test_fp16_round_up_is_smallest_upper_neighbour():
    pos = np.arange(1, 0x7C00, dtype=np.uint16)          # every positive finite fp16
    vals = pos.view(np.float16).astype(np.float64)
    # an exact fp16 value rounds up to itself
    for b, v in zip(pos[::7], vals[::7]):
        assert oracle.fp16_round_up(v) == b
    # just above a value -> the next fp16 (or saturation at the top)
    for b, v in zip(pos[::13], vals[::13]):
        up = oracle.fp16_round_up(np.nextafter(v, np.inf))
        assert up == (b + 1 if b < 0x7BFF else 0x7BFF)
    # random reals: result >= x and its predecessor < x
    r = np.random.default_rng(1)
    xs = np.concatenate([10.0 ** r.uniform(-9, 4.8, 4000), r.uniform(0, 1e-7, 200)])
    for x in xs[xs > 0]:
        h = oracle.fp16_round_up(x)
        hv = float(np.uint16(h).view(np.float16))
        assert hv >= x
        if h > 1:
            assert float(np.uint16(h - 1).view(np.float16)) < x
    assert oracle.fp16_round_up(1e-30) == 1                # smallest subnormal
    assert oracle.fp16_round_up(70000.0) == 0x7BFF         # saturation reading


def test_rne_encoders_vs_libraries():
    r = np.random.default_rng(2)
    xs = np.concatenate([r.standard_normal(3000) * 10.0 ** r.integers(-6, 4, 3000),
                         [0.0, -0.0, 1.0, -2.5, 65504.0, 6e-8, 3e-5]])
    for x in xs:
        assert oracle.round_to_dtype_bits(x, "fp16") == int(np.float16(x).view(np.uint16))
    # bf16: use float32-exact inputs and exact halfway points so that torch's
    # conversion path cannot double-round.
    f32 = (r.standard_normal(3000) * 10.0 ** r.integers(-20, 20, 3000)).astype(np.float32)
    for x in f32.astype(np.float64):
        ref = int(torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16)) & 0xFFFF
        assert oracle.round_to_dtype_bits(x, "bf16") == ref
    # halfway between 1.0 (0x3F80) and next (0x3F81) -> even (0x3F80); 0x3F81/0x3F82 -> 0x3F82
    assert oracle.round_to_dtype_bits(1.0 + 2.0 ** -8, "bf16") == 0x3F80
    assert oracle.round_to_dtype_bits(1.0 + 3 * 2.0 ** -8, "bf16") == 0x3F82


# ---------------------------------------------------------------- quantizer
def _rows(dtype, n, D, seed, std=1.0):
    r = np.random.default_rng(seed)
    x = (r.standard_normal((n, D)) * std).astype(np.float32)
    return W.to_bits(x, dtype)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("std", [1.0, 0.5, 20.0, 1e-3])
def test_quantizer_page_facts(dtype, std):
    x = _rows(dtype, 400, 128, 3, std)
    x[5] = 0                                             # an all-zero token
    x[7, 3] = 0                                          # an exact zero element
    q, s = oracle.quantize_rows(x, dtype)
    xd = oracle.bits_to_double(x, dtype)
    sd = oracle.bits_to_double(s, "fp16")
    # codes within [-127, 127]; never -128
    assert q.min() >= FACTS["code_min"] and q.max() <= FACTS["code_max"]
    assert not np.any(q == -128)
    # exact zero -> code 0, dequantized exactly 0
    assert np.all(q[xd == 0.0] == FACTS["zero_code"])
    assert np.all(q[xd == 0.0].astype(np.float64) * np.broadcast_to(sd[:, None], q.shape)[xd == 0.0] == 0.0)
    # element error bound
    err = np.abs(xd - q.astype(np.float64) * sd[:, None])
    assert np.all(err <= sd[:, None] / 2 + FACTS["error_slack"])
    # all-zero token -> scale 1.0 and all codes 0
    assert s[5] == int(FACTS["zero_token_scale_bits"]) and np.all(q[5] == 0)
    # the largest-magnitude coordinate maps to +-127 whenever the scale is normal
    a = np.abs(xd).max(axis=1)
    normal = (sd >= 2.0 ** -14) & (a > 0)
    amax = np.abs(xd).argmax(axis=1)
    codes = q[np.arange(len(q)), amax]
    assert np.all(np.abs(codes[normal]) == FACTS["max_coordinate_code"])
    # odd symmetry: q(-x) = -q(x)
    qn, sn = oracle.quantize_rows(x ^ np.uint16(0x8000), dtype)
    assert np.array_equal(sn, s) and np.array_equal(qn, -q)


def test_scale_is_absmax_over_127_rounded_up_exactly():
    """Exact rational check: s >= a/127 and the previous fp16 is < a/127."""
    for dtype in ("fp16", "bf16"):
        x = _rows(dtype, 300, 64, 4, 1.0)
        x[:50] = _rows(dtype, 50, 64, 5, 1e-4)       # pushes scales into fp16 subnormals
        _, s = oracle.quantize_rows(x, dtype)
        for row, sb in zip(x, s):
            a = max(Fraction(abs(v)) for v in oracle.bits_to_double(row, dtype))
            sv = Fraction(float(np.uint16(sb).view(np.float16)))
            assert sv >= a / FACTS["scale_divisor"].__int__()
            if sb > 1:
                prev = Fraction(float(np.uint16(sb - 1).view(np.float16)))
                assert prev < a / 127


def test_quantizer_brute_force_band_exact_rounding():
    """For fixed scales, every fp16 x of a band is rounded exactly like the
    rational x/s with ties to even (fractions + Python's round, which is
    round-half-even)."""
    for sb in (0x3C00, 0x2409, 0x1E66, 0x0003):       # 1.0, ~0.01576, ~0.0062, subnormal
        s = Fraction(float(np.uint16(sb).view(np.float16)))
        limit = float(127 * s)
        band = np.arange(0, 0x7C00, 3, dtype=np.uint16)
        vals = band.view(np.float16).astype(np.float64)
        band = band[vals <= limit]
        for bits in (band, band | np.uint16(0x8000)):
            q = oracle.quantize_row(bits, "fp16", sb)
            for b, c in zip(bits, q):
                ref = round(Fraction(float(np.uint16(b).view(np.float16))) / s)
                assert c == max(-127, min(127, ref))


def test_quantizer_exact_ties_round_to_even():
    # s = 1.0: x = 2.5 -> 2, 3.5 -> 4, -0.5 -> 0, 126.5 -> 126
    row = np.array([2.5, 3.5, -0.5, 126.5, 127.0, 0.5, 1.5, -2.5], dtype=np.float16).view(np.uint16)
    s = oracle.token_scale(row, "fp16")
    assert s == 0x3C00                                   # a = 127 -> exactly 1.0
    assert list(oracle.quantize_row(row, "fp16", s)) == [2, 4, 0, 126, 127, 0, 2, -2]


def test_mlxcel_scale_floor_bug_is_caught():
    """Planting the scale-floor defect described on the mlxcel page (the scale
    clamped to at least 1.0) in the oracle's quantizer breaks the +-127 fact
    that the pins above enforce."""
    x = _rows("bf16", 50, 128, 6, 1.0)
    xd = oracle.bits_to_double(x, "bf16")
    hits = 0
    for row, rd in zip(x, xd):
        s = oracle.token_scale(row, "bf16")
        s_bug = max(s, 0x3C00)                            # the planted mistake
        q_bug = oracle.quantize_row(row, "bf16", s_bug)
        hits += int(abs(q_bug[np.abs(rd).argmax()]) == 127)
    assert hits == 0


def test_scale_saturation_reading():
    big = W.f32_to_bf16_bits(np.array([1e7, -3.0, 2e7, 0.0], dtype=np.float32))
    s = oracle.token_scale(big, "bf16")
    assert s == 0x7BFF
    q = oracle.quantize_row(big, "bf16", s)
    assert list(q) == [127, 0, 127, 0]


# -------------------------------------------------------------- page bytes
def test_page_bytes_match_page_figure():
    with open(os.path.join(GOLDEN, "page_bytes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for bs, hk, d, b8, b16, ratio in rows:
        bs, hk, d, b8, b16 = map(int, (bs, hk, d, b8, b16))
        assert oracle.page_bytes_int8(bs, hk, d) == b8
        assert oracle.page_bytes_native16(bs, hk, d) == b16
        assert b8 / b16 == float(ratio)


# --------------------------------------------------------------- paging
def test_quantize_append_places_rows_by_slot():
    w = W.make("tiny")
    nb, bt, _ = w.tables()
    Hkv, D, bs = w.num_kv_heads, w.head_dim, w.block_size
    kc = np.zeros((nb, Hkv, bs, D), np.int8); vc = np.zeros_like(kc)
    ks = np.zeros((nb, Hkv, bs), np.uint16); vs = np.zeros_like(ks)
    for b in range(w.num_seqs):
        k, v = w.seq_kv(b)
        L = len(k)
        slots = w.slots(b, 0, L)
        slots[3] = -1                                    # skipped token
        bad = oracle.quantize_append(k, v, "fp16", slots, kc, vc, ks, vs, bs)
        assert bad == 0
        qk, sk = oracle.quantize_rows(k, "fp16")
        qv, sv = oracle.quantize_rows(v, "fp16")
        for t in range(L):
            blk, off = bt[b, t // bs], t % bs
            if t == 3:
                assert np.all(kc[blk, :, off] == 0) and np.all(ks[blk, :, off] == 0)
                continue
            assert np.array_equal(kc[blk, :, off], qk[t]) and np.array_equal(vc[blk, :, off], qv[t])
            assert np.array_equal(ks[blk, :, off], sk[t]) and np.array_equal(vs[blk, :, off], sv[t])
    bad = oracle.quantize_append(k[:2], v[:2], "fp16", np.array([nb * bs, -5]), kc, vc, ks, vs, bs)
    assert bad == 1


# -------------------------------------------------------------- attention
def _sdpa_ref(qd, kd, vd, sm_scale):
    """torch float64 SDPA, GQA by consecutive grouping (repeat_interleave)."""
    Hq, Hkv = qd.shape[0], kd.shape[1]
    q = torch.from_numpy(qd)[None, :, None, :]
    k = torch.from_numpy(np.ascontiguousarray(kd.transpose(1, 0, 2)))[None]
    v = torch.from_numpy(np.ascontiguousarray(vd.transpose(1, 0, 2)))[None]
    k = k.repeat_interleave(Hq // Hkv, dim=1)
    v = v.repeat_interleave(Hq // Hkv, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=sm_scale)
    return o[0, :, 0, :].numpy()


@pytest.mark.parametrize("L,Hq,Hkv,D,dtype", [(17, 4, 2, 64, "fp16"), (40, 4, 2, 64, "fp16"),
                                              (33, 8, 2, 128, "bf16"), (5, 3, 3, 64, "bf16"),
                                              (64, 8, 1, 128, "fp16")])
def test_decode_matches_torch_sdpa(L, Hq, Hkv, D, dtype):
    w = W.custom(1, Hq, Hkv, D, dtype, [L], seed=L)
    k, v = w.seq_kv(0)
    q = w.seq_q(0)
    for quantized in (True, False):
        out, bits = oracle.decode_sequence(q, k, v, dtype, w.sm_scale, quantized=quantized)
        if quantized:
            qk, sk = oracle.quantize_rows(k, dtype)
            qv, sv = oracle.quantize_rows(v, dtype)
            kd = qk.astype(np.float64) * oracle.bits_to_double(sk, "fp16")[..., None]
            vd = qv.astype(np.float64) * oracle.bits_to_double(sv, "fp16")[..., None]
        else:
            kd, vd = oracle.bits_to_double(k, dtype), oracle.bits_to_double(v, dtype)
        ref = _sdpa_ref(oracle.bits_to_double(q, dtype), kd, vd, w.sm_scale)
        np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
        ref_bits = np.array([[oracle.round_to_dtype_bits(x, dtype) for x in r] for r in out])
        assert np.array_equal(bits, ref_bits)


def test_single_token_context_returns_v():
    w = W.custom(1, 4, 2, 64, "fp16", [1], seed=11)
    k, v = w.seq_kv(0)
    out, _ = oracle.decode_sequence(w.seq_q(0), k, v, "fp16", w.sm_scale)
    qv, sv = oracle.quantize_rows(v, "fp16")
    vhat = qv[0].astype(np.float64) * oracle.bits_to_double(sv[0], "fp16")[:, None]
    for h in range(4):
        assert np.array_equal(out[h], vhat[h // 2])


def test_equal_keys_return_mean_of_v():
    w = W.custom(1, 4, 2, 64, "bf16", [23], seed=12)
    k, v = w.seq_kv(0)
    k[:] = k[0]                                          # every key identical
    out, _ = oracle.decode_sequence(w.seq_q(0), k, v, "bf16", w.sm_scale)
    qv, sv = oracle.quantize_rows(v, "bf16")
    vhat = qv.astype(np.float64) * oracle.bits_to_double(sv, "fp16")[..., None]
    mean = vhat.mean(axis=0)
    for h in range(4):
        np.testing.assert_allclose(out[h], mean[h // 2], rtol=0, atol=1e-14)


def test_partitioned_combine_equals_direct():
    r = np.random.default_rng(7)
    for L in (1, 15, 16, 17, 300, 1000):
        q = r.standard_normal(64); k = r.standard_normal((L, 64)) * 3; v = r.standard_normal((L, 64))
        ref = oracle.attend_one(q, k, v, 0.125)
        for part in (1, 7, 16, 256, 4096):
            np.testing.assert_allclose(oracle.attend_one(q, k, v, 0.125, partition=part), ref,
                                       rtol=0, atol=1e-12)


def test_zero_length_context_is_zero():
    out = oracle.attend_one(np.ones(64), np.zeros((0, 64)), np.zeros((0, 64)), 0.125)
    assert np.all(out == 0.0)


def test_sampled_heads_match_full_decode():
    w = W.custom(1, 8, 2, 64, "bf16", [50], seed=13)
    k, v = w.seq_kv(0)
    q = w.seq_q(0)
    full, fb = oracle.decode_sequence(q, k, v, "bf16", w.sm_scale)
    part, pb = oracle.decode_sequence(q, k, v, "bf16", w.sm_scale, heads=[7, 0, 5])
    assert np.array_equal(part, full[[7, 0, 5]]) and np.array_equal(pb, fb[[7, 0, 5]])


def test_dequantize_rows_vs_library_rounding():
    """Dequantize-window baseline: code * scale rounded once to the dtype,
    against numpy's float16 and torch's bfloat16 conversions of the exact
    product (both round to nearest even), including overflow to inf and the
    signs of zero."""
    r = np.random.default_rng(11)
    N, D = 64, 32
    codes = r.integers(-127, 128, size=(N, D)).astype(np.int8)
    codes[0, :4] = [0, 127, -127, 1]
    scales = r.integers(0x0001, 0x7C00, size=N).astype(np.uint16)   # finite positive fp16
    scales[:3] = [0x7BFF, 0x0001, 0x3C00]                          # 65504, min subnormal, 1
    exact = codes.astype(np.float64) * np.array(
        [oracle.fp16_to_double(int(s)) for s in scales])[:, None]
    got16 = oracle.dequantize_rows(codes, scales, "fp16")
    with np.errstate(over="ignore"):                              # 127 * 65504 overflows
        want16 = exact.astype(np.float16).view(np.uint16)
    assert np.array_equal(got16, want16)
    assert got16[0, 1] == 0x7C00 and got16[0, 2] == 0xFC00          # 127 * 65504 -> +-inf
    gotbf = oracle.dequantize_rows(codes, scales, "bf16")
    wantbf = torch.from_numpy(exact).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gotbf, wantbf)
    # a wrong row/scale pairing (transposed operand) must not pass: scales differ by row
    assert not np.array_equal(oracle.dequantize_rows(codes, scales[::-1].copy(), "fp16"), want16)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("scale", [1.0, 0.05, 0.0371, 3.5e-4])
def test_static_quantizer_vs_float32_arithmetic(dtype, scale):
    """Static per-tensor scale: against numpy's IEEE float32 reciprocal and
    product, round half to even, clamp; plus the error bound inside the range,
    odd symmetry and the default scale 1.0 (codes = rounded values)."""
    r = np.random.default_rng(int(scale * 1e4) + len(dtype))
    x = (r.standard_normal((200, 64)) * 127 * scale * 0.4).astype(np.float32)
    x[0, :6] = [0.0, 127 * scale, -127 * scale, 300 * scale, -300 * scale, 2.5 * scale]
    if dtype == "fp16":
        bits = x.astype(np.float16).view(np.uint16)
        xv = bits.view(np.float16).astype(np.float32)
    else:
        bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        xv = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    s32 = np.float32(scale)
    inv = np.float32(1.0) / s32
    want = np.clip(np.rint(xv * inv), -127, 127).astype(np.int8)      # float32 product, RNE
    got = oracle.quantize_rows_static(bits, dtype, scale)
    assert np.array_equal(got, want)
    assert got.min() >= -127
    inside = np.abs(xv.astype(np.float64)) <= 126 * float(s32)
    err = np.abs(xv.astype(np.float64) - got.astype(np.float64) * float(s32))
    # the fp32 reciprocal and product move x/s by at most ~2^-23 relative, so a
    # value within that of a half step may round across it: s/2 (1 + 1e-4)
    assert np.all(err[inside] <= float(s32) / 2 * (1 + 1e-4))
    neg = bits ^ np.uint16(0x8000)
    assert np.array_equal(oracle.quantize_rows_static(neg, dtype, scale), -got)
    if scale == 1.0:
        assert np.array_equal(got, np.clip(np.rint(xv), -127, 127).astype(np.int8))


def test_static_scale_quality_below_tokenwise_when_token_norms_vary():
    """The comparison the static variant exists for: when token magnitudes
    vary (log-normal norms, sigma 1 -- large tokens such as attention sinks
    next to many small ones), one calibrated per-tensor scale (max|x| / 127
    over the tensor, as the static-scale pages calibrate) resolves the small
    tokens far more coarsely than one scale per token: the dequantized K/V
    error is several times larger, and so is the attention error against the
    unquantized values (seeded case)."""
    r = np.random.default_rng(17)
    L, Hkv, G, D = 512, 2, 4, 128
    sm = 1.0 / np.sqrt(D)

    def bf16(x):
        return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(
            torch.int16).numpy().view(np.uint16)
    norms = np.exp(1.0 * r.standard_normal((L, Hkv, 1)))
    k = bf16(r.standard_normal((L, Hkv, D)) * norms)
    v = bf16(r.standard_normal((L, Hkv, D)) * norms)
    q = bf16(r.standard_normal((Hkv * G, D)))
    kf, vf, qf = (oracle.bits_to_double(a, "bf16") for a in (k, v, q))
    # element level: relative RMS error of the dequantized tensors
    def rel_rms(xf, xh):
        return np.sqrt(np.mean((xh - xf) ** 2) / np.mean(xf ** 2))
    ck, sck = oracle.quantize_rows(k, "bf16")
    kt = ck.astype(np.float64) * oracle.bits_to_double(sck, "fp16")[..., None]
    sk = float(np.float32(np.abs(kf).max() / 127))
    sv = float(np.float32(np.abs(vf).max() / 127))
    kh = oracle.quantize_rows_static(k, "bf16", sk).astype(np.float64) * sk
    vh = oracle.quantize_rows_static(v, "bf16", sv).astype(np.float64) * sv
    assert rel_rms(kf, kh) > 3 * rel_rms(kf, kt)
    # attention level
    exact, _ = oracle.decode_sequence(q, k, v, "bf16", sm, quantized=False)
    tok, _ = oracle.decode_sequence(q, k, v, "bf16", sm, quantized=True)
    st = np.stack([oracle.attend_one(qf[h], kh[:, h // G], vh[:, h // G], sm)
                   for h in range(Hkv * G)])
    err_tok = np.abs(tok - exact).max()
    err_static = np.abs(st - exact).max()
    assert err_static > 2 * err_tok, (err_static, err_tok)


def test_trim_keep_sink_matches_page_examples_and_composes():
    """Front trim keeping the sink: the kept positions of the worked cases in
    tests/golden/trim_keep_sink.txt (from the page's rule: [first keep] ++
    [the rest after the next n], exactly n removed, keep = 0 the old front
    trim, clamped to the sequence); trimming n1 then n2 equals trimming
    n1 + n2 with the same keep; rows (payload or scale rows) move intact."""
    with open(os.path.join(GOLDEN, "trim_keep_sink.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            L, keep, n, kept = [x.strip() for x in line.split("|")]
            L, keep, n = int(L), int(keep), int(n)
            pos = np.arange(L, dtype=np.int64)
            got = oracle.trim_keep_sink(pos, keep, n)
            assert got.tolist() == [int(x) for x in kept.split()], (L, keep, n)
    r = np.random.default_rng(3)
    rows = r.integers(-127, 128, size=(300, 8, 16)).astype(np.int8)
    for keep in (0, 4, 17):
        for n1, n2 in ((5, 9), (1, 1), (100, 150)):
            two = oracle.trim_keep_sink(oracle.trim_keep_sink(rows, keep, n1), keep, n2)
            one = oracle.trim_keep_sink(rows, keep, n1 + n2)
            assert np.array_equal(two, one)
            assert len(one) == 300 - (n1 + n2)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_prefill_matches_causal_torch_sdpa_and_decode(dtype):
    """Chunked prefill: against torch's float64 scaled_dot_product_attention
    with a causal mask offset by the cached prefix (GQA by repeat), over the
    native values; its last query row equals the decode of the whole
    sequence; a chunk of one query is the decode."""
    r = np.random.default_rng(23)
    L, n, Hkv, G, D = 70, 19, 2, 3, 64
    Hq = Hkv * G
    if dtype == "fp16":
        mk = lambda *s: r.standard_normal(s).astype(np.float16).view(np.uint16)  # noqa: E731
    else:
        mk = lambda *s: torch.from_numpy(r.standard_normal(s).astype(np.float32)).to(  # noqa: E731
            torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    k, v, q = mk(L, Hkv, D), mk(L, Hkv, D), mk(n, Hq, D)
    sm = 0.11
    out, _ = oracle.prefill_sequence(q, k, v, dtype, sm, quantized=False)
    qt = torch.from_numpy(oracle.bits_to_double(q, dtype)).permute(1, 0, 2)       # [Hq, n, D]
    kt = torch.from_numpy(oracle.bits_to_double(k, dtype)).permute(1, 0, 2).repeat_interleave(G, 0)
    vt = torch.from_numpy(oracle.bits_to_double(v, dtype)).permute(1, 0, 2).repeat_interleave(G, 0)
    pos = torch.arange(L - n, L)[:, None]
    mask = torch.arange(L)[None, :] <= pos                                         # [n, L]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=sm)
    assert np.allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    outq, _ = oracle.prefill_sequence(q, k, v, dtype, sm, quantized=True)
    dec, _ = oracle.decode_sequence(q[-1], k, v, dtype, sm, quantized=True)
    assert np.allclose(outq[-1], dec, rtol=0, atol=1e-13)
    one, _ = oracle.prefill_sequence(q[:1], k[:L - n + 1], v[:L - n + 1], dtype, sm)
    dec1, _ = oracle.decode_sequence(q[0], k[:L - n + 1], v[:L - n + 1], dtype, sm)
    assert np.allclose(one[0], dec1, rtol=0, atol=1e-13)
