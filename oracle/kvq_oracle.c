/*
 * FP64 CPU oracle for tokenwise symmetric INT8 KV-cache quantization and
 * dequantized decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker of the CUDA
 * library; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code, header, table or helper with the CUDA path.
 *
 * Plain, slow, obviously-correct loops in double precision.  No blocking, no
 * fusion, no reordering beyond what each definition states.
 *
 * Sources (page title, then section):
 *  [MI] "feat: opt-in INT8 KV-cache quantization" (MoE-Infinity PR #183),
 *       "What landed" and "Precision & memory": one FP16 scale per
 *       (layer, page, KV head, token), rounded upward; symmetric, no -128,
 *       exact zero, element error <= stored_scale/2 + 1e-6; INT8 payload plus
 *       FP16 scale per page; decode dequantizes and accumulates in FP32 and is
 *       checked against an FP32 dequantized softmax-attention oracle.
 *  [ML] "fix(cuda/kv): correct Int8 KV per-token scale ..." (mlxcel PR #717),
 *       "The Int8 bug and fix": scale = absmax/127, replaced by 1.0 only for an
 *       all-zero token; the max-magnitude coordinate then maps to +-127.
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes of the repository):
 *  - rounding of x/s to an integer: round half to even;
 *  - "rounded upward": the smallest FP16 value h with 127*h >= absmax;
 *  - absmax/127 above the largest finite FP16 (65504): the scale saturates to
 *    65504 and the codes clamp to +-127 (out of contract: error bound void);
 *  - cache layout: payload [num_blocks][num_kv_heads][block_size][head_dim]
 *    int8, scale plane [num_blocks][num_kv_heads][block_size] FP16 bits;
 *    slot = block * block_size + offset, slot < 0 means "skip";
 *  - GQA: query head h reads KV head h / (Hq / Hkv);
 *  - attention output rounded once, round-to-nearest-even, to the dtype of q.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_FP16_MAX_BITS 0x7BFFu /* 65504 */
#define ORC_FP16_ONE_BITS 0x3C00u /* 1.0 */

/* ---------------------------------------------------------------------------
 * IEEE binary16 / bfloat16 <-> double, from the format definitions.
 * ------------------------------------------------------------------------- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_fp16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = (m == 0) ? INFINITY : NAN;
  else
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

double orc_bits_to_double(uint16_t bits, int is_bf16) {
  return is_bf16 ? orc_bf16_to_double(bits) : orc_fp16_to_double(bits);
}

/* Encode a non-negative finite x on the binary16 grid with the integer
 * significand chosen by `round_fn` (ceil or rint).  Exponent e is the binade of
 * x, floored at -14 (the subnormals share the step of the lowest binade). */
static uint16_t fp16_encode_nonneg(double x, double (*round_fn)(double)) {
  if (x == 0.0) return 0;
  int E;
  frexp(x, &E); /* x in [2^(E-1), 2^E) */
  int e = E - 1;
  if (e < -14) e = -14;
  double step = ldexp(1.0, e - 10);
  double m = round_fn(x / step); /* division by a power of two: exact */
  /* value = m * step with m in [0, 2048]; the bit pattern is continuous across
   * the subnormal/normal boundary and across a carry into the next binade. */
  long bits = ((long)(e + 15) << 10) + (long)m - 1024;
  if (bits >= 0x7C00) return 0x7C00; /* overflow -> +inf */
  return (uint16_t)bits;
}

/* Smallest binary16 value >= x, for finite x > 0; saturates at 65504. */
uint16_t orc_fp16_round_up(double x) {
  if (x > 65504.0) return ORC_FP16_MAX_BITS;
  return fp16_encode_nonneg(x, ceil);
}

/* Round-to-nearest-even double -> binary16 (for attention outputs). */
uint16_t orc_fp16_from_double_rne(double x) {
  if (isnan(x)) return 0x7E00;
  uint16_t s = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isinf(a)) return s | 0x7C00;
  return s | fp16_encode_nonneg(a, rint); /* rint: current mode, RNE */
}

/* Round-to-nearest-even double -> bfloat16 (8-bit significand, exponent bias
 * 127, subnormal step 2^-133). */
uint16_t orc_bf16_from_double_rne(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t s = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isinf(a)) return s | 0x7F80;
  if (a == 0.0) return s;
  int E;
  frexp(a, &E);
  int e = E - 1;
  if (e < -126) e = -126;
  double step = ldexp(1.0, e - 7);
  double m = rint(a / step);
  long bits = ((long)(e + 127) << 7) + (long)m - 128;
  if (bits >= 0x7F80) return s | 0x7F80;
  return s | (uint16_t)bits;
}

uint16_t orc_from_double_rne(double x, int is_bf16) {
  return is_bf16 ? orc_bf16_from_double_rne(x) : orc_fp16_from_double_rne(x);
}

/* ---------------------------------------------------------------------------
 * Quantizer [MI] "What landed", [ML] "The Int8 bug and fix".
 * ------------------------------------------------------------------------- */

/* Per-token scale of one (token, KV head) row of D elements:
 *   a = max_d |x_d|;  s = 1.0 if a == 0, else the smallest FP16 h with
 *   127 * h >= a  (that is, absmax/127 rounded upward to FP16).
 * 127*h is exact in double (11 + 7 significant bits), so the defining
 * inequality is checked exactly; the division only seeds the search. */
uint16_t orc_token_scale(const uint16_t* row, int D, int is_bf16) {
  double a = 0.0;
  for (int d = 0; d < D; ++d) {
    double x = fabs(orc_bits_to_double(row[d], is_bf16));
    if (x > a) a = x;
  }
  if (a == 0.0) return ORC_FP16_ONE_BITS; /* all-zero token [ML] */
  if (a > 127.0 * 65504.0) return ORC_FP16_MAX_BITS; /* saturation reading */
  uint16_t h = orc_fp16_round_up(a / 127.0);
  /* exact fix-up on the definition (positive binary16 bits are monotone) */
  while (h > 1 && 127.0 * orc_fp16_to_double((uint16_t)(h - 1)) >= a) --h;
  while (127.0 * orc_fp16_to_double(h) < a) ++h;
  return h;
}

/* Codes of one row for a given scale s:
 *   q_d = clamp(round_half_even(x_d / s), -127, 127).
 * x and s are exact in double and an exact tie x/s = k + 1/2 is exactly
 * representable, so rint() on the double quotient is the exact rounding. */
void orc_quantize_row(const uint16_t* row, int D, int is_bf16,
                      uint16_t scale_bits, int8_t* q) {
  double s = orc_fp16_to_double(scale_bits);
  for (int d = 0; d < D; ++d) {
    double r = rint(orc_bits_to_double(row[d], is_bf16) / s);
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    q[d] = (int8_t)r;
  }
}

/* Dequantized value of a code: s * q (exact in double). */
double orc_dequant(int8_t q, uint16_t scale_bits) {
  return orc_fp16_to_double(scale_bits) * (double)q;
}

/* Dequantize-window baseline ([ML] "The Int8 bug and fix": its CUDA path
 * dequantizes the whole cached window to the activation dtype, then runs
 * SDPA): every code times its row's scale, rounded once (round to nearest
 * even) to the dtype.  codes [N][D], scales [N] -> out [N][D] dtype bits. */
void orc_dequantize_rows(const int8_t* q, const uint16_t* scales, int64_t N, int D,
                         int is_bf16, uint16_t* out) {
  for (int64_t n = 0; n < N; ++n)
    for (int d = 0; d < D; ++d)
      out[n * D + d] = orc_from_double_rne(orc_dequant(q[n * D + d], scales[n]), is_bf16);
}

/* Static (per-tensor) scale quantizer: "fix: #552 int8 kv cache quantization
 * cannot be enabled" (InfiniLM PR #553) -- one static scale per tensor
 * (default 1.0, or calibrated from max|K| / 127); "Add calibrated INT8 KV
 * cache to PyTorch backend" (TensorRT-LLM PR #18953) -- a calibrated scalar
 * (shared by K and V) applied through its reciprocal.  Reading: the scale s
 * is binary32, inv = fl32(1 / s), and
 *   q = clamp(round_half_even(fl32(x * inv)), -127, 127)
 * (the code format of the tokenwise path, no -128).  x * inv is exact in
 * double (at most 11 + 24 significant bits), so converting it to float is
 * the single fp32 rounding of the definition. */
void orc_quantize_rows_static(const uint16_t* x, int64_t N, int D, int is_bf16, float s,
                              int8_t* q) {
  const float inv = 1.0f / s;
  for (int64_t i = 0; i < N * (int64_t)D; ++i) {
    const float p = (float)(orc_bits_to_double(x[i], is_bf16) * (double)inv);
    double r = rint((double)p);
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    q[i] = (int8_t)r;
  }
}

/* Front trim that keeps the attention sink: "fix(cuda/kv): correct Int8 KV
 * per-token scale ..." (mlxcel PR #717) follow-up commit, "The fix" -- with
 * keep > 0 the sequence becomes [first keep tokens] ++ [the rest after the
 * next n], exactly n tokens removed, the INT8 payload and its scales sliced
 * in lockstep; keep = 0 is the plain front trim.  Reading: keep and n are
 * clamped to the sequence (keep <= L, n <= L - keep).  Rows are `row_bytes`
 * bytes (one token's payload, or its scale row); in [L] -> out [L'] with
 * L' = L - n returned. */
int64_t orc_trim_keep_sink(const uint8_t* in, int64_t L, int64_t row_bytes, int64_t keep,
                           int64_t n, uint8_t* out) {
  if (keep < 0) keep = 0;
  if (keep > L) keep = L;
  if (n < 0) n = 0;
  if (n > L - keep) n = L - keep;
  int64_t o = 0;
  for (int64_t t = 0; t < L; ++t) {
    if (t >= keep && t < keep + n) continue;             /* the n tokens after the sink */
    memcpy(out + o * row_bytes, in + t * row_bytes, (size_t)row_bytes);
    ++o;
  }
  return o;
}

/* Quantize rows [N][D] into codes [N][D] and scales [N]. */
void orc_quantize_rows(const uint16_t* x, int64_t N, int D, int is_bf16,
                       int8_t* q, uint16_t* scales) {
  for (int64_t n = 0; n < N; ++n) {
    scales[n] = orc_token_scale(x + n * D, D, is_bf16);
    orc_quantize_row(x + n * D, D, is_bf16, scales[n], q + n * D);
  }
}

/* Quantize-on-write of T new tokens into the paged cache.
 *   k, v: [T][Hkv][D] with a row stride of `k_token_stride` / `v_token_stride`
 *         elements between consecutive tokens (heads contiguous, stride D);
 *   slot_mapping[t]: -1 (or any negative) skips token t; otherwise the token
 *         lands at block = slot / bs, offset = slot % bs.
 * Writes payload [NB][Hkv][bs][D] and scale plane [NB][Hkv][bs].
 * Returns the number of tokens whose slot was out of range (not written). */
int64_t orc_quantize_append(const uint16_t* k, const uint16_t* v,
                            int64_t k_token_stride, int64_t v_token_stride,
                            int64_t T, int Hkv, int D, int is_bf16,
                            const int64_t* slot_mapping, int8_t* k_cache,
                            int8_t* v_cache, uint16_t* k_scale,
                            uint16_t* v_scale, int64_t num_blocks, int bs) {
  int64_t bad = 0;
  for (int64_t t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * bs) {
      ++bad;
      continue;
    }
    int64_t blk = slot / bs, off = slot % bs;
    for (int j = 0; j < Hkv; ++j) {
      int64_t row = (blk * Hkv + j) * bs + off; /* [NB][Hkv][bs] index */
      const uint16_t* kr = k + t * k_token_stride + (int64_t)j * D;
      const uint16_t* vr = v + t * v_token_stride + (int64_t)j * D;
      k_scale[row] = orc_token_scale(kr, D, is_bf16);
      v_scale[row] = orc_token_scale(vr, D, is_bf16);
      orc_quantize_row(kr, D, is_bf16, k_scale[row], k_cache + row * D);
      orc_quantize_row(vr, D, is_bf16, v_scale[row], v_cache + row * D);
    }
  }
  return bad;
}

/* ---------------------------------------------------------------------------
 * Decode attention over dequantized tokens ([MI] "What landed": dequantized
 * SDPA oracle; GQA head sharing).
 * ------------------------------------------------------------------------- */

/* One sequence, one query head, L tokens of one KV head, given as dequantized
 * (or native-precision) values k_hat, v_hat: [L][row_stride] with the head's D
 * values at offset 0 of each row.
 *   z_t = sm_scale * sum_d q_d * k_t,d ;  p = softmax(z) ;  out = sum_t p_t v_t
 * For L == 0 the output is zero (reading). */
void orc_attend_one(const double* q, const double* k_hat, const double* v_hat,
                    int64_t L, int64_t row_stride, int D, double sm_scale,
                    double* out) {
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (L <= 0) return;
  double zmax = -INFINITY;
  for (int64_t t = 0; t < L; ++t) {
    double z = 0.0;
    for (int d = 0; d < D; ++d) z += q[d] * k_hat[t * row_stride + d];
    z *= sm_scale;
    if (z > zmax) zmax = z;
  }
  double denom = 0.0;
  for (int64_t t = 0; t < L; ++t) {
    double z = 0.0;
    for (int d = 0; d < D; ++d) z += q[d] * k_hat[t * row_stride + d];
    double p = exp(z * sm_scale - zmax);
    denom += p;
    for (int d = 0; d < D; ++d) out[d] += p * v_hat[t * row_stride + d];
  }
  for (int d = 0; d < D; ++d) out[d] /= denom;
}

/* The same attention evaluated in partitions of `part` tokens, each giving a
 * local max m_i, sum l_i = sum exp(z - m_i) and o_i = sum exp(z - m_i) v, then
 * merged by  M = max m_i,  L = sum l_i e^(m_i-M),  out = sum o_i e^(m_i-M) / L.
 * Algebraically identical to orc_attend_one for any partition size; used to
 * pin the split-K combine rule. */
void orc_attend_one_partitioned(const double* q, const double* k_hat,
                                const double* v_hat, int64_t L,
                                int64_t row_stride, int D, double sm_scale,
                                int64_t part, double* out, double* scratch) {
  /* scratch: D doubles */
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (L <= 0) return;
  double M = -INFINITY, Lsum = 0.0;
  for (int64_t t0 = 0; t0 < L; t0 += part) {
    int64_t t1 = t0 + part < L ? t0 + part : L;
    double mi = -INFINITY;
    for (int64_t t = t0; t < t1; ++t) {
      double z = 0.0;
      for (int d = 0; d < D; ++d) z += q[d] * k_hat[t * row_stride + d];
      z *= sm_scale;
      if (z > mi) mi = z;
    }
    double li = 0.0;
    for (int d = 0; d < D; ++d) scratch[d] = 0.0;
    for (int64_t t = t0; t < t1; ++t) {
      double z = 0.0;
      for (int d = 0; d < D; ++d) z += q[d] * k_hat[t * row_stride + d];
      double p = exp(z * sm_scale - mi);
      li += p;
      for (int d = 0; d < D; ++d) scratch[d] += p * v_hat[t * row_stride + d];
    }
    /* merge (m_i, l_i, o_i) into the running (M, Lsum, out) */
    double Mn = mi > M ? mi : M;
    double a_old = exp(M - Mn), a_new = exp(mi - Mn);
    Lsum = Lsum * a_old + li * a_new;
    for (int d = 0; d < D; ++d) out[d] = out[d] * a_old + scratch[d] * a_new;
    M = Mn;
  }
  for (int d = 0; d < D; ++d) out[d] /= Lsum;
}

/* Full decode of one sequence from its own unpaged token arrays.
 *   q: [Hq][D] bits;  k, v: [L][Hkv][D] bits (the tokens as written);
 *   quantized = 1: each (token, KV head) row is quantized with the oracle's
 *   own quantizer and dequantized (s * q) before attention; quantized = 0:
 *   the native 16-bit values are used (reference for the 16-bit twin).
 *   out: [Hq][D] doubles (unrounded);  out_bits: [Hq][D] rounded (RNE) to
 *   the dtype of q, may be NULL.
 *   heads: if non-NULL, only the listed query heads (n_heads of them) are
 *   computed, in that order, into out[i][D].
 * work: 2 * L * D doubles + L * D int8 + D doubles of caller scratch. */
void orc_decode_sequence(const uint16_t* q, const uint16_t* k,
                         const uint16_t* v, int64_t L, int Hq, int Hkv, int D,
                         int is_bf16, int quantized, double sm_scale,
                         const int32_t* heads, int n_heads, double* out,
                         uint16_t* out_bits, double* work, int8_t* qwork) {
  int G = Hq / Hkv;
  double* k_hat = work;
  double* v_hat = work + L * (int64_t)D;
  int nh = heads ? n_heads : Hq;
  int cur_j = -1;
  for (int i = 0; i < nh; ++i) {
    int h = heads ? heads[i] : i;
    int j = h / G;
    if (j != cur_j) { /* (re)build the dequantized rows of KV head j */
      for (int64_t t = 0; t < L; ++t) {
        const uint16_t* kr = k + (t * Hkv + j) * (int64_t)D;
        const uint16_t* vr = v + (t * Hkv + j) * (int64_t)D;
        if (quantized) {
          uint16_t sk = orc_token_scale(kr, D, is_bf16);
          uint16_t sv = orc_token_scale(vr, D, is_bf16);
          orc_quantize_row(kr, D, is_bf16, sk, qwork);
          for (int d = 0; d < D; ++d) k_hat[t * D + d] = orc_dequant(qwork[d], sk);
          orc_quantize_row(vr, D, is_bf16, sv, qwork);
          for (int d = 0; d < D; ++d) v_hat[t * D + d] = orc_dequant(qwork[d], sv);
        } else {
          for (int d = 0; d < D; ++d) {
            k_hat[t * D + d] = orc_bits_to_double(kr[d], is_bf16);
            v_hat[t * D + d] = orc_bits_to_double(vr[d], is_bf16);
          }
        }
      }
      cur_j = j;
    }
    double qd[256];
    for (int d = 0; d < D; ++d) qd[d] = orc_bits_to_double(q[(int64_t)h * D + d], is_bf16);
    orc_attend_one(qd, k_hat, v_hat, L, D, D, sm_scale, out + (int64_t)i * D);
    if (out_bits)
      for (int d = 0; d < D; ++d)
        out_bits[(int64_t)i * D + d] = orc_from_double_rne(out[(int64_t)i * D + d], is_bf16);
  }
}

/* Chunked prefill over the same cache: "fix(cuda/kv): correct Int8 KV
 * per-token scale ..." (mlxcel PR #717), "Server integration" -- Int8
 * chunked prefill + decode.  Reading: the n query tokens of the chunk are the
 * last n of the sequence's L tokens (already written), and query i (position
 * p = L - n + i) attends causally to tokens 0..p:
 *   out[i][h] = softmax_t<=p(sm_scale * q[i][h] . k_hat_t) . v_hat
 * q: [n][Hq][D]; k, v: [L][Hkv][D]; out, out_bits: [n][Hq][D].  work holds
 * 2 * L * D doubles (dequantized rows of one KV head at a time). */
void orc_prefill_sequence(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t L,
                          int64_t n, int Hq, int Hkv, int D, int is_bf16, int quantized,
                          double sm_scale, double* out, uint16_t* out_bits, double* work,
                          int8_t* qwork) {
  int G = Hq / Hkv;
  double* k_hat = work;
  double* v_hat = work + L * (int64_t)D;
  for (int j = 0; j < Hkv; ++j) {
    for (int64_t t = 0; t < L; ++t) {
      const uint16_t* kr = k + (t * Hkv + j) * (int64_t)D;
      const uint16_t* vr = v + (t * Hkv + j) * (int64_t)D;
      if (quantized) {
        uint16_t sk = orc_token_scale(kr, D, is_bf16);
        uint16_t sv = orc_token_scale(vr, D, is_bf16);
        orc_quantize_row(kr, D, is_bf16, sk, qwork);
        for (int d = 0; d < D; ++d) k_hat[t * D + d] = orc_dequant(qwork[d], sk);
        orc_quantize_row(vr, D, is_bf16, sv, qwork);
        for (int d = 0; d < D; ++d) v_hat[t * D + d] = orc_dequant(qwork[d], sv);
      } else {
        for (int d = 0; d < D; ++d) {
          k_hat[t * D + d] = orc_bits_to_double(kr[d], is_bf16);
          v_hat[t * D + d] = orc_bits_to_double(vr[d], is_bf16);
        }
      }
    }
    for (int64_t i = 0; i < n; ++i) {
      const int64_t len = L - n + i + 1;              /* tokens 0..p */
      for (int g = 0; g < G; ++g) {
        const int h = j * G + g;
        double qd[256];
        const int64_t row = (i * Hq + h) * (int64_t)D;
        for (int d = 0; d < D; ++d) qd[d] = orc_bits_to_double(q[row + d], is_bf16);
        orc_attend_one(qd, k_hat, v_hat, len, D, D, sm_scale, out + row);
        if (out_bits)
          for (int d = 0; d < D; ++d) out_bits[row + d] = orc_from_double_rne(out[row + d], is_bf16);
      }
    }
  }
}

/* Bytes of one cache page in the two layouts ([MI] "Precision & memory"):
 *   INT8: K and V payload (1 byte per element) + one FP16 scale per
 *         (KV head, token) for K and for V;
 *   native 16-bit: K and V at 2 bytes per element. */
int64_t orc_page_bytes_int8(int bs, int Hkv, int D) {
  return 2LL * bs * Hkv * D * 1 + 2LL * bs * Hkv * 2;
}
int64_t orc_page_bytes_native16(int bs, int Hkv, int D) {
  return 2LL * bs * Hkv * D * 2;
}
