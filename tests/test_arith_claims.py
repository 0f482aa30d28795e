"""Exhaustive CPU checks of the bit-level arithmetic the kernels rely on.

- INT8 code -> FP16 without a conversion instruction: the code's byte XOR
  0x80 (its offset-binary form u = c + 128) is placed under the exponent byte
  0x64, giving the FP16 value 1024 + u; subtracting 1152 (0x6480) leaves c.
  Both steps are exact for every byte, and a code's FP16 value is an integer
  the tensor cores multiply exactly.
- bf16 -> FP16 for the queries: every bf16 value whose magnitude lies in
  FP16's normal range [2^-14, 65504] is representable in FP16 (8 significant
  bits into 11), so the rounding to FP16 is exact there.
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
