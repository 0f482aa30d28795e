"""Exhaustive CPU checks of the bit-level arithmetic the kernels rely on.

- INT8 code -> FP16 without a conversion instruction: the code's byte XOR
  0x80 (its offset-binary form u = c + 128) is placed under the exponent byte
  0x64, giving the FP16 value 1024 + u; subtracting 1152 (0x6480) leaves c.
  Both steps are exact for every byte, and a code's FP16 value is an integer
  the tensor cores multiply exactly.
- bf16 -> FP16 for the queries: every bf16 value whose magnitude lies in
  FP16's normal range [2^-14, 65504] is representable in FP16 (8 significant
  bits into 11), so the rounding to FP16 is exact there.
- Outside FP16's normal range the BF16 queries are first multiplied by a
  power of two 2^-sh chosen from the largest magnitude of the row (or head):
  it lands in [2^14, 2^15), so nothing overflows, and every element within
  2^-28 of that magnitude is still exact in FP16.
- The tokenwise V scales multiply the softmax weights, not the codes:
  P' = p * s_v * 2^-E with E the exponent of the largest scale seen (FP16
  biased exponent in the decode, FP32 in the prefill) stays below 2 (times
  the prefill's 2^8 lazy-rescale slack), far inside FP16, for every FP16
  scale, where code * s_v itself can exceed 65504.
- The quantizer rounds x / s half to even without a division: k = rint(x
  times an approximate reciprocal of s) is within one of the answer, the
  remainder x - k s is exact in one FMA, and its comparison with s / 2 (ties
  to the even neighbour) gives the answer; checked for every fp16 and bf16
  value against scales from the smallest subnormal to 65504.
- The static-scale decode folds the K scale into the score scale and the V
  scale into the output; the tokenwise one multiplies the scale after the
  integer dot product: both are re-associations of the same product, checked
  here on random data in FP64 as the identity they are."""
import numpy as np


def test_int8_to_fp16_byte_trick_is_exact_for_every_code():
    codes = np.arange(-128, 128, dtype=np.int16)
    byte = codes.astype(np.int8).view(np.uint8).astype(np.uint16)
    biased = (np.uint16(0x64) << 8) | (byte ^ np.uint16(0x80))
    v = biased.view(np.float16).astype(np.float64)
    assert np.array_equal(v, 1024.0 + codes + 128)              # 1024 + u, u = c + 128
    bias = np.array([0x6480], dtype=np.uint16).view(np.float16)[0]
    assert float(bias) == 1152.0
    out = (biased.view(np.float16) - bias).astype(np.float64)   # FP16 subtraction
    assert np.array_equal(out, codes.astype(np.float64))
    # the pair layout the kernels use: bytes 0, 1 -> halves of one word, 2, 3 -> the next
    word = np.array([0x80FF017F], dtype=np.uint32)              # bytes 0x7F, 0x01, 0xFF, 0x80
    b = word.view(np.uint8)
    assert list(b.astype(np.int8)) == [127, 1, -1, -128]


def test_bf16_to_fp16_exact_in_normal_range():
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    f32 = (bits << 16).view(np.float32)
    with np.errstate(invalid="ignore"):
        a = np.abs(f32.astype(np.float64))
    normal = np.isfinite(a) & (a >= 2.0 ** -14) & (a <= 65504.0)
    h = f32[normal].astype(np.float16)
    assert np.array_equal(h.astype(np.float64), f32[normal].astype(np.float64))
    assert normal.sum() == 2 * 30 * 128        # both signs, exponents -14..15, 7-bit mantissas


def test_scale_folding_is_a_reassociation():
    r = np.random.default_rng(3)
    q = r.standard_normal(64)
    codes = r.integers(-127, 128, size=(16, 64)).astype(np.float64)
    s = r.uniform(0.001, 0.1, size=16)
    sm = 0.125
    direct = sm * (q[None, :] * (s[:, None] * codes)).sum(1)     # dequantize, then dot
    folded = (sm * s) * (codes @ q)                               # integer dot, then scale
    assert np.allclose(direct, folded, rtol=1e-13, atol=0)


def _bf16_fp16_shift(max_bits: np.ndarray) -> np.ndarray:
    """The kernels' shift: biased BF16 exponent - 127 - 14, kept in [-126, 113]."""
    return np.clip((max_bits >> 7).astype(np.int64) - 141, -126, 113)


def test_bf16_query_shift_maps_the_maximum_into_fp16_and_keeps_near_elements_exact():
    bits = np.arange(1, 0x7F80, dtype=np.uint32)                  # positive finite BF16
    x = (bits << 16).view(np.float32).astype(np.float64)
    sh = _bf16_fp16_shift(bits)
    y = x * 2.0 ** (-sh)
    unclamped = (bits >> 7).astype(np.int64) - 141 >= -126          # normal maxima
    assert np.all((y[unclamped] >= 2.0 ** 14) & (y[unclamped] < 2.0 ** 15))
    assert np.all(y <= 65504.0)                                     # never overflows FP16
    # every element of the row is exact in FP16 unless it is below 2^-14 after
    # the shift, i.e. 2^28 times smaller than the row's maximum
    for m in (0x3F80, 0x4780, 0x4B7D, 0x3380, 0x7F7F, 0x0080):      # 1, 65536, ~1.7e7, ...
        shm = int(_bf16_fp16_shift(np.array([m], np.uint32))[0])
        xs = x[bits <= m] * 2.0 ** (-shm)
        ok = xs >= 2.0 ** -14
        assert np.array_equal(xs[ok].astype(np.float16).astype(np.float64), xs[ok])
        assert np.all(x[bits <= m][~ok] < x[bits == m][0] * 2.0 ** -27)


def test_v_scale_on_p_stays_inside_fp16():
    s_bits = np.arange(1, 0x7C00, dtype=np.uint16)                  # every positive FP16 scale
    s = s_bits.view(np.float16).astype(np.float64)
    assert s.max() == 65504.0
    # decode: E = max(FP16 biased exponent, 1); p <= 1
    e16 = np.maximum(s_bits >> 10, 1).astype(np.int64)
    r16 = s * 2.0 ** (15 - e16)
    assert np.all((r16 < 2.0)) and np.all(r16[s_bits >= 0x0400] >= 1.0)
    # the running maximum only grows, so every earlier scale is below it too
    # prefill: E = FP32 biased exponent of the scale; p <= 2^8 between rescales
    e32 = (s.astype(np.float32).view(np.uint32) >> 23).astype(np.int64)
    r32 = s * 2.0 ** (127 - e32)
    assert np.all((r32 >= 1.0) & (r32 < 2.0))
    assert 2.0 ** 8 * r32.max() < 65504.0
    # where the old formulation overflowed: 127 * s rounded to FP16
    with np.errstate(over="ignore"):
        big = (127.0 * s).astype(np.float16)
    assert np.isinf(big).sum() > 0 and not np.isinf(r16.astype(np.float16)).any()



def _quant_code_f32(x, s, inv, sat=True):
    """The quantizer's division-free code, step by step in float32: q = x *
    inv limited to +-256, k = rint(q) by adding 1.5 * 2^23 (k read back as an
    integer from the sum's bits), the remainder x - k s (one FMA: exact while
    |k| <= 128), one step towards the exact quotient's round-half-even
    neighbour, and the clamp to +-127."""
    x = x.astype(np.float32)
    s, inv = np.float32(s), np.float32(inv)
    q = (x * inv).astype(np.float32)
    if sat:                                   # a saturated scale: the quotient may pass 127
        q = np.clip(q, -256, 256).astype(np.float32)
    big = np.float32(12582912.0)
    t = (q + big).astype(np.float32)
    k = (t - big).astype(np.float32)
    ki = t.view(np.uint32).astype(np.int64) - 0x4B400000
    r64 = x.astype(np.float64) - k.astype(np.float64) * np.float64(s)
    inb = np.abs(k) <= 128
    assert np.all(r64[inb].astype(np.float32).astype(np.float64) == r64[inb])   # FMA exact
    r = r64.astype(np.float32)
    h = np.float32(0.5) * s
    odd = (ki & 1) != 0
    ki = ki + ((r > h) | ((r == h) & odd)) - ((r < -h) | ((r == -h) & odd))
    return np.clip(ki, -127, 127) if sat else ki


def test_quantizer_rounding_without_division_is_exact():
    # every finite fp16 and bf16 value against FP16 scales from subnormal to
    # saturated, with the reciprocal off by up to two ulp (the kernel takes an
    # approximate one)
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    f16 = bits.astype(np.uint16).view(np.float16).astype(np.float32)
    b16 = (bits << 16).view(np.float32)
    scales = [np.float16(v) for v in (2.0 ** -24, 2.0 ** -14, 0.0372, 0.5, 1.0, 3.0, 258.0,
                                      4097.0, 65504.0)]
    for xs in (f16, b16):
        xs = xs[np.isfinite(xs)]
        for sc in scales:
            s = np.float32(sc)
            want = np.clip(np.rint(xs.astype(np.float64) / np.float64(s)), -127, 127)
            for ulps in (-2, 0, 2):
                inv = np.float32(1) / s
                for _ in range(abs(ulps)):
                    inv = np.nextafter(inv, np.float32(np.inf if ulps > 0 else -np.inf),
                                       dtype=np.float32)
                with np.errstate(over="ignore", invalid="ignore"):
                    got = _quant_code_f32(xs, s, inv)
                assert np.array_equal(got, want), (float(s), ulps)
                # an unsaturated scale bounds the row's quotients by 127: no clamps
                inside = np.abs(xs.astype(np.float64)) <= 127 * np.float64(s)
                got = _quant_code_f32(xs[inside], s, inv, sat=False)
                assert np.array_equal(got, want[inside]), (float(s), ulps, "unsaturated")


def _quant_fast_f32(x, s, ulps=0):
    """The quantizer's fast path for an unsaturated row, step by step in
    float32: inv = 1/s off by `ulps` ulp, k = rint(x * inv) (the product
    rounded, then the integer by adding 1.5 * 2^23), and the tie flag
    |x - k s| == s/2 from the exact remainder."""
    x = x.astype(np.float32)
    s = np.float32(s)
    inv = np.float32(1) / s
    for _ in range(abs(ulps)):
        inv = np.nextafter(inv, np.float32(np.inf if ulps > 0 else -np.inf), dtype=np.float32)
    q = (x * inv).astype(np.float32)
    big = np.float32(12582912.0)
    t = (q + big).astype(np.float32)
    k = (t - big).astype(np.float32)
    ki = t.view(np.uint32).astype(np.int64) - 0x4B400000
    r64 = x.astype(np.float64) - k.astype(np.float64) * np.float64(s)
    assert np.all(r64.astype(np.float32).astype(np.float64) == r64)   # FMA exact
    tie = np.abs(r64) == 0.5 * np.float64(s)
    return ki, tie


def _row_scale_f32(a):
    """The row scale's FP16 bits, step by step in float32: y = a * fl(1/127),
    rounded up to FP16, saturated at 65504, then one step down when 127 times
    the FP16 value below still covers a."""
    a = a.astype(np.float32)
    y = (a * np.float32(1.0 / 127.0)).astype(np.float32)
    with np.errstate(over="ignore"):
        rn = y.astype(np.float16)
    bits = rn.view(np.uint16).astype(np.int64) + (rn.astype(np.float32) < y)
    sat = bits >= 0x7C00
    below = np.clip(bits - 1, 0, 0x7BFF).astype(np.uint16).view(np.float16).astype(np.float32)
    down = (np.float32(127.0) * below).astype(np.float32) >= a
    return np.where(sat, 0x7BFF, bits - (down & ~sat))


def test_row_scale_without_division_is_exact():
    # every positive finite fp16 and bf16 magnitude: the division-free scale
    # equals a/127 rounded up to FP16 (saturated at 65504), decided in float64
    bits = np.arange(1, 1 << 15, dtype=np.uint32)
    f16 = bits.astype(np.uint16).view(np.float16).astype(np.float32)
    b16 = (bits << 16).view(np.float32)
    for a in (f16, b16):
        a = a[np.isfinite(a)]
        q = a.astype(np.float64) / 127.0
        with np.errstate(over="ignore"):
            rn = q.astype(np.float16)
        want = rn.view(np.uint16).astype(np.int64) + (rn.astype(np.float64) < q)
        want = np.where(want >= 0x7C00, 0x7BFF, want)
        assert np.array_equal(_row_scale_f32(a), want)
        assert np.all(want >= 1)


def test_quantizer_fast_path_is_exact_off_ties():
    # every finite fp16 and bf16 value of an unsaturated row (|x| <= 127 s)
    # against 600 FP16 scales (subnormal to 65504, a seeded sample plus the
    # edges), the reciprocal off by up to two ulp: the fast code equals the exact quotient's round-half-even code
    # wherever the remainder does not flag a tie, and every flagged element is
    # an exact tie (|x/s - k| = 1/2 exactly)
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    f16 = bits.astype(np.uint16).view(np.float16).astype(np.float32)
    b16 = (bits << 16).view(np.float32)
    rng = np.random.default_rng(7)
    pats = np.concatenate([rng.integers(1, 0x7BFF, 580), [1, 2, 0x03FF, 0x0400, 0x3C00, 0x3C01,
                                                          0x2008, 0x5BF0, 0x7800, 0x7BFE, 0x7BFF,
                                                          0x0001, 0x1C00, 0x3555, 0x4B00,
                                                          0x57F0, 0x6000, 0x6400, 0x7000, 0x77FF]])
    ties = 0
    for xs in (f16, b16):
        xs = xs[np.isfinite(xs)]
        for pat in pats:
            s = np.float32(np.uint16(pat).view(np.float16))
            sub = xs[np.abs(xs.astype(np.float64)) <= 127 * np.float64(s)]
            want = np.rint(sub.astype(np.float64) / np.float64(s)).astype(np.int64)
            for ulps in (-2, 0, 2):                  # the kernel's reciprocal is approximate
                ki, tie = _quant_fast_f32(sub, s, ulps)
                assert np.all(tie | (ki == want)), (float(s), ulps)
                k64 = ki.astype(np.float64)
                assert np.all(np.abs(sub[tie].astype(np.float64) / np.float64(s) - k64[tie]) == 0.5)
                ties += int(tie.sum())
    assert ties > 0                              # the tie branch is exercised
