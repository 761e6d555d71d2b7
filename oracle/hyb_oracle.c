/*
 * hyb_oracle.c -- float64 CPU oracle for the DeepSeek-V4 hybrid-attention forward
 * (CSA + HCA + sliding window).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: it exists so that tests, the smoke check and the CPU-baseline leg
 * of the benchmark can compare the CUDA library against a plain, slow, obviously
 * correct restatement of the method.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * Style rules kept on purpose:
 *   - single thread, plain loops, no BLAS, no blocking, no fusion;
 *   - all arithmetic in double, except the FP8 quantiser, whose integer decision
 *     (the code) is taken in float32 exactly as the kernel takes it;
 *   - every input is decoded to double by this file's own decoders, written
 *     from the number-format definitions (bf16 = top half of an IEEE binary32;
 *     e4m3 = 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 *     infinities, S.1111.111 = NaN, largest finite 448).
 *
 * Sources (web pages on DeepSeek-V4):
 *   [HA]  "DeepSeek-V4 hybrid attention: CSA, HCA, mHC, MoE" (trishampatil.com),
 *         sections IV (RMSNorm, partial RoPE and attention sink inside both
 *         branches), V.1 (compression with overlap), V.2 (lightning indexer),
 *         V.3 (core attention), VI (HCA).
 *   [DV4] "DeepSeek-V4: Anatomy of an Open-Source Frontier Model"
 *         (modernaiengineering.com), "One query in a CSA layer",
 *         csa_hca_budget.py and the worked example "three formulas".
 *   [KE]  "DeepSeek-V4 Architecture From Kernels" (shivasnotes.com),
 *         section 9 (heterogeneous KV cache: tails, window).
 *   [MA]  "Mastering DeepSeek-V4 Architecture, Course 1" (mailtotanvir.github.io),
 *         model configurations table.
 *   [JH]  PyTorch walkthrough re-posted on juhe.plus, "The Code: RoPE Helpers"
 *         (rotary convention: consecutive pairs, frequencies theta^(-2i/d)).
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes of the repository):
 *   R1 gates are per channel: S = softmax over the window positions of
 *      (Z + positional bias), taken separately for each channel ([HA] V.1,
 *      "element-wise product").
 *   R2 CSA entry i pools stream a over block i and stream b over block i-1 in
 *      ONE softmax over all 2m logits ([HA] V.1 prose "block i-1 and block i").
 *   R3 entry 0 has no block -1: its stream-b logits are -inf, so it is a
 *      softmax over its m stream-a rows only.
 *   R4 positional bias is [2m][c] for CSA (row 0 = first token of block i-1,
 *      row 2m-1 = last token of block i) and [m'][c] for HCA.
 *   R5 causality: an entry is visible to query position t only when its last
 *      token is <= t, i.e. s < floor((t+1)/m) ([HA] V.2 "preceding blocks";
 *      unfinished tails are covered by the window, [KE] section 9).
 *   R6 top-k keeps min(k, visible) entries ranked by (score desc, index asc),
 *      returned sorted by ascending entry index and padded with -1
 *      ([DV4] worked example: "top-k cannot pick more entries than exist").
 *   R7 an empty attended set gives o = 0 and lse = -inf.
 *   R8 the window branch attends raw rows max(0, t-n_win+1) .. t and is merged
 *      with the compressed branch as one softmax over the union multiset
 *      ([DV4] step 5 "ordinary attention over about 1,152 entries").
 *   R9 FP8 scaling: one float32 scale per row = amax/448 (1 when amax = 0);
 *      code = round-to-nearest-even of x/scale, saturated to +-448.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype codes understood by this file (its own numbering) */
#define ORC_F32 0
#define ORC_BF16 1
#define ORC_E4M3 2

/* ---------------------------------------------------------------- formats */

/* bf16: the upper 16 bits of an IEEE-754 binary32. */
double orc_bf16_decode(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &bits, 4);
  return (double)f;
}

/* e4m3 (OCP FP8): sign(1) exponent(4, bias 7) mantissa(3); exponent field 0 is
 * subnormal (0.mmm * 2^-6); S.1111.111 is NaN; no infinities. */
double orc_e4m3_decode(uint8_t v) {
  int sign = (v >> 7) & 1;
  int e = (v >> 3) & 0xF;
  int mant = v & 7;
  double mag;
  if (e == 15 && mant == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)mant / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)mant / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* Nearest e4m3 code to a float32 value, ties to the even code, saturating to
 * +-448 (the "satfinite" convention).  Written as a brute-force search over
 * the 127 non-negative finite codes so that it is correct by inspection. */
uint8_t orc_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  double ax = fabs((double)x);
  int best = 0;
  double best_err = INFINITY;
  for (int code = 0; code <= 0x7E; ++code) {
    double err = fabs(orc_e4m3_decode((uint8_t)code) - ax);
    if (err < best_err || (err == best_err && (code & 1) == 0)) {
      best = code;
      best_err = err;
    }
  }
  if (ax > 448.0) best = 0x7E; /* saturate */
  return (uint8_t)((x < 0 || (x == 0 && signbit(x))) ? (best | 0x80) : best);
}

/* Round a double to the nearest bf16 value (ties to even), returned as double.
 * bf16 keeps 8 significant bits, the binary32 exponent range, and subnormals
 * spaced 2^-133 apart.  Used only to build the oracle's own end-to-end chain
 * (entries stored in bf16). */
double orc_round_bf16(double x) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e;
  frexp(x, &e);               /* |x| = f * 2^e, f in [0.5, 1) */
  int q = e - 8;              /* spacing exponent for 8 significant bits */
  if (q < -133) q = -133;     /* subnormal spacing */
  double r = nearbyint(ldexp(x, -q)); /* default rounding mode: to nearest even */
  double y = ldexp(r, q);
  if (fabs(y) > 3.3895313892515355e38) /* beyond largest finite bf16 -> inf */
    y = copysign(INFINITY, x);
  return y;
}

static double load_elem(int dtype, const void* p, int64_t i) {
  switch (dtype) {
    case ORC_F32: return (double)((const float*)p)[i];
    case ORC_BF16: return orc_bf16_decode(((const uint16_t*)p)[i]);
    case ORC_E4M3: return orc_e4m3_decode(((const uint8_t*)p)[i]);
  }
  return NAN;
}

/* ------------------------------------------------------------- counting */

/* Number of entries written for n_rows input rows starting at absolute block
 * first_block: one per complete block, except that with overlap a first block
 * other than block 0 only serves as the previous block of the next one. */
int64_t orc_compress_out_count(int64_t n_rows, int64_t m, int overlap, int64_t first_block) {
  int64_t blocks = n_rows / m;
  int64_t skip = (overlap && first_block > 0) ? 1 : 0;
  return blocks > skip ? blocks - skip : 0;
}

/* Entries visible to query position t (reading R5). */
int64_t orc_visible(int64_t t, int64_t m) { return (t + 1) / m; }

/* Window rows attended by query position t (reading R8). */
int64_t orc_window_count(int64_t t, int64_t n_win) { return t + 1 < n_win ? t + 1 : n_win; }

/* --------------------------------------------------------------- compress */

/*
 * Softmax-gated compressor ([HA] V.1 for CSA with overlap, [HA] VI for HCA).
 *
 * Inputs: ca/za (stream a values and gating logits) and, when overlap = 1,
 * cb/zb (stream b), all [B][n_rows][c] of dtype `dtype`; bias [P][c] float32
 * with P = 2m (overlap) or m.  Row r of the inputs is absolute token
 * first_block*m + r.  Output: out [B][n_out][c] double, n_out from
 * orc_compress_out_count; output j is absolute entry first_block + j (+1 when
 * the first block is only a previous block).
 *
 * For entry i and channel ch the window holds (overlap) the m stream-b rows of
 * block i-1 at positions 0..m-1 and the m stream-a rows of block i at positions
 * m..2m-1 (HCA: the m stream-a rows of block i at positions 0..m-1).  Logit of
 * a row = Z[row][ch] + bias[position][ch]; S = softmax over the window; the
 * entry is sum over the window of S * C[row][ch].
 */
void orc_compress(int dtype, const void* ca, const void* cb, const void* za, const void* zb,
                  const float* bias, int64_t B, int64_t n_rows, int64_t c, int64_t m, int overlap,
                  int64_t first_block, double* out) {
  int64_t n_out = orc_compress_out_count(n_rows, m, overlap, first_block);
  int64_t skip = (overlap && first_block > 0) ? 1 : 0;
  int64_t P = overlap ? 2 * m : m;
  double* logit = (double*)malloc(sizeof(double) * (size_t)P);
  double* val = (double*)malloc(sizeof(double) * (size_t)P);
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t j = 0; j < n_out; ++j) {
      int64_t lb = j + skip;              /* local block index of stream a */
      int64_t abs_blk = first_block + lb; /* absolute block index */
      for (int64_t ch = 0; ch < c; ++ch) {
        int64_t np = 0;
        if (overlap) {
          /* positions 0..m-1: stream b over block i-1 (absent for block 0) */
          for (int64_t p = 0; p < m; ++p) {
            if (abs_blk == 0) {
              logit[np] = -INFINITY;
              val[np] = 0.0;
            } else {
              int64_t row = (lb - 1) * m + p;
              int64_t off = (b * n_rows + row) * c + ch;
              logit[np] = load_elem(dtype, zb, off) + (double)bias[p * c + ch];
              val[np] = load_elem(dtype, cb, off);
            }
            ++np;
          }
        }
        /* stream a over block i */
        for (int64_t p = 0; p < m; ++p) {
          int64_t row = lb * m + p;
          int64_t off = (b * n_rows + row) * c + ch;
          int64_t pos = overlap ? m + p : p;
          logit[np] = load_elem(dtype, za, off) + (double)bias[pos * c + ch];
          val[np] = load_elem(dtype, ca, off);
          ++np;
        }
        double mx = -INFINITY;
        for (int64_t p = 0; p < np; ++p)
          if (logit[p] > mx) mx = logit[p];
        double den = 0.0, num = 0.0;
        for (int64_t p = 0; p < np; ++p) {
          if (logit[p] == -INFINITY) continue;
          double e = exp(logit[p] - mx);
          den += e;
          num += e * val[p];
        }
        out[(b * n_out + j) * c + ch] = num / den;
      }
    }
  }
  free(logit);
  free(val);
}

/* The pooling weights themselves, for the sum-to-one invariant: weights
 * [P] for one (batch, output entry, channel), same window layout as above. */
void orc_compress_weights(int dtype, const void* za, const void* zb, const float* bias, int64_t n_rows,
                          int64_t c, int64_t m, int overlap, int64_t first_block, int64_t b, int64_t j,
                          int64_t ch, double* weights) {
  int64_t skip = (overlap && first_block > 0) ? 1 : 0;
  int64_t P = overlap ? 2 * m : m;
  int64_t lb = j + skip, abs_blk = first_block + lb;
  double* logit = (double*)malloc(sizeof(double) * (size_t)P);
  int64_t np = 0;
  if (overlap) {
    for (int64_t p = 0; p < m; ++p) {
      if (abs_blk == 0)
        logit[np++] = -INFINITY;
      else
        logit[np++] = load_elem(dtype, zb, (b * n_rows + (lb - 1) * m + p) * c + ch) + (double)bias[p * c + ch];
    }
  }
  for (int64_t p = 0; p < m; ++p) {
    int64_t pos = overlap ? m + p : p;
    logit[np++] = load_elem(dtype, za, (b * n_rows + lb * m + p) * c + ch) + (double)bias[pos * c + ch];
  }
  double mx = -INFINITY, den = 0.0;
  for (int64_t p = 0; p < np; ++p)
    if (logit[p] > mx) mx = logit[p];
  for (int64_t p = 0; p < np; ++p) den += (logit[p] == -INFINITY) ? 0.0 : exp(logit[p] - mx);
  for (int64_t p = 0; p < np; ++p) weights[p] = (logit[p] == -INFINITY) ? 0.0 : exp(logit[p] - mx) / den;
  free(logit);
}

/* -------------------------------------------------------------- quantise */

/* Row-wise FP8 quantiser (reading R9).  Decisions in float32, as the kernel
 * takes them: amax = max |x| (exact), scale = amax / 448 (IEEE division),
 * code = orc_e4m3_encode(x / scale) (IEEE division). */
void orc_quantise_fp8_rows(const float* x, int64_t rows, int64_t c, uint8_t* codes, float* scales) {
  for (int64_t r = 0; r < rows; ++r) {
    float amax = 0.0f;
    for (int64_t ch = 0; ch < c; ++ch) {
      float a = fabsf(x[r * c + ch]);
      if (a > amax) amax = a;
    }
    volatile float scale = (amax > 0.0f) ? amax / 448.0f : 1.0f;
    scales[r] = scale;
    for (int64_t ch = 0; ch < c; ++ch) {
      volatile float y = x[r * c + ch] / scale;
      codes[r * c + ch] = orc_e4m3_encode(y);
    }
  }
}

/* -------------------------------------------------------------- MXFP4
 * FP4 for the indexer's query-key path ("DeepSeek-V4: Anatomy..." (modernaiengineering.com),
 * "FP4 quantization-aware training": V4 applies FP4 to the indexer's query-key path).
 * The pages name no format; the OCP microscaling one is taken (reading R23): e2m1
 * elements in blocks of 32 sharing one e8m0 power-of-two scale.
 */

/* e2m1: sign(1) exponent(2, bias 1) mantissa(1); exponent field 0 is subnormal
 * (0.m * 2^0); no infinities or NaN; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_decode(uint8_t v) {
  int sign = (v >> 3) & 1;
  int e = (v >> 1) & 3;
  int mant = v & 1;
  double mag = (e == 0) ? 0.5 * (double)mant : ldexp(1.0 + 0.5 * (double)mant, e - 1);
  return sign ? -mag : mag;
}

/* e8m0: 2^(e - 127); e = 255 is NaN. */
double orc_e8m0_decode(uint8_t e) { return e == 255 ? NAN : ldexp(1.0, (int)e - 127); }

/* Nearest e2m1 code, ties to the even code, saturating to +-6 (brute force over
 * the 8 non-negative codes). */
uint8_t orc_e2m1_encode(float x) {
  double ax = fabs((double)x);
  int best = 0;
  double best_err = INFINITY;
  for (int code = 0; code <= 7; ++code) {
    double err = fabs(orc_e2m1_decode((uint8_t)code) - ax);
    if (err < best_err || (err == best_err && (code & 1) == 0)) {
      best = code;
      best_err = err;
    }
  }
  if (ax > 6.0) best = 7;
  return (uint8_t)((x < 0 || (x == 0 && signbit(x))) ? (best | 8) : best);
}

/* Rows of c values (c a multiple of 32) to MXFP4: per block of 32, the shared
 * exponent E = floor(log2(amax)) - 2 (2 = the exponent of e2m1's largest
 * magnitude, 6 = 1.5 * 2^2), clamped to [-127, 127] (E = -127 when amax = 0);
 * scale code E + 127; element code = e2m1 of x / 2^E (exact: a power of two).
 * codes [rows][c] (one code per byte), scales [rows][c/32]. */
void orc_quantise_mxfp4_rows(const float* x, int64_t rows, int64_t c, uint8_t* codes, uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b0 = 0; b0 < c; b0 += 32) {
      float amax = 0.0f;
      for (int64_t i = b0; i < b0 + 32; ++i) {
        float a = fabsf(x[r * c + i]);
        if (a > amax) amax = a;
      }
      int E = -127;
      if (amax > 0.0f) {
        int e;
        frexp((double)amax, &e); /* amax = f * 2^e, f in [0.5, 1): floor(log2 amax) = e - 1 */
        E = (e - 1) - 2;
        if (E < -127) E = -127;
        if (E > 127) E = 127;
      }
      scales[r * (c / 32) + b0 / 32] = (uint8_t)(E + 127);
      for (int64_t i = b0; i < b0 + 32; ++i) codes[r * c + i] = orc_e2m1_encode((float)ldexp((double)x[r * c + i], -E));
    }
}

/* ------------------------------------------------------- lightning indexer */

/*
 * Index scores ([HA] V.2):  I[t,s] = sum_h w[t,h] * ReLU(q_I[t,h] . K_I[s]),
 * for the entries s < floor((t+1)/m) (reading R5); others are set to -inf.
 *
 * qI [B][n_q][n_ih][c_I] and kI [B][N][c_I] of dtype qk_dtype (F32 or E4M3);
 * with E4M3 the decoded codes are multiplied by qI_scale [B][n_q][n_ih] and
 * kI_scale [B][N].  w [B][n_q][n_ih] float32.  Query j sits at absolute
 * position q_pos0 + j.  Output scores [B][n_q][N] double.
 */
void orc_index_scores(int qk_dtype, const void* qI, const float* qI_scale, const float* w, const void* kI,
                      const float* kI_scale, int64_t B, int64_t n_q, int64_t N, int64_t n_ih, int64_t c_I,
                      int64_t m, int64_t q_pos0, double* scores) {
  double* qd = (double*)malloc(sizeof(double) * (size_t)(n_ih * c_I));
  double* kd = (double*)malloc(sizeof(double) * (size_t)c_I);
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t j = 0; j < n_q; ++j) {
      int64_t t = q_pos0 + j;
      int64_t vis = orc_visible(t, m);
      for (int64_t h = 0; h < n_ih; ++h) {
        double sq = (qk_dtype == ORC_E4M3) ? (double)qI_scale[(b * n_q + j) * n_ih + h] : 1.0;
        for (int64_t d = 0; d < c_I; ++d)
          qd[h * c_I + d] = load_elem(qk_dtype, qI, ((b * n_q + j) * n_ih + h) * c_I + d) * sq;
      }
      for (int64_t s = 0; s < N; ++s) {
        double* dst = &scores[(b * n_q + j) * N + s];
        if (s >= vis) {
          *dst = -INFINITY;
          continue;
        }
        double sk = (qk_dtype == ORC_E4M3) ? (double)kI_scale[b * N + s] : 1.0;
        for (int64_t d = 0; d < c_I; ++d) kd[d] = load_elem(qk_dtype, kI, (b * N + s) * c_I + d) * sk;
        double acc = 0.0;
        for (int64_t h = 0; h < n_ih; ++h) {
          double dot = 0.0;
          for (int64_t d = 0; d < c_I; ++d) dot += qd[h * c_I + d] * kd[d];
          double relu = dot > 0.0 ? dot : 0.0;
          acc += (double)w[(b * n_q + j) * n_ih + h] * relu;
        }
        *dst = acc;
      }
    }
  }
  free(qd);
  free(kd);
}

/* ------------------------------------------------------------------ top-k */

typedef struct {
  double score;
  int64_t index;
} orc_scored;

static int cmp_rank(const void* a, const void* b) {
  const orc_scored* x = (const orc_scored*)a;
  const orc_scored* y = (const orc_scored*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->index < y->index) ? -1 : (x->index > y->index);
}

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/*
 * Top-k selector ([HA] V.2 "keeps the highest-scoring blocks"; reading R6).
 * scores [rows][N]; visible[r] = number of leading entries row r may see.
 * idx [rows][k] receives min(k, visible[r]) entry indices sorted ascending,
 * padded with -1.  Ranking: score descending, then index ascending.
 */
void orc_topk(const double* scores, const int64_t* visible, int64_t rows, int64_t N, int64_t k, int32_t* idx) {
  orc_scored* buf = (orc_scored*)malloc(sizeof(orc_scored) * (size_t)(N > 0 ? N : 1));
  for (int64_t r = 0; r < rows; ++r) {
    int64_t v = visible[r] < N ? visible[r] : N;
    for (int64_t s = 0; s < v; ++s) {
      buf[s].score = scores[r * N + s];
      buf[s].index = s;
    }
    qsort(buf, (size_t)v, sizeof(orc_scored), cmp_rank);
    int64_t take = v < k ? v : k;
    int32_t* out = &idx[r * k];
    for (int64_t i = 0; i < take; ++i) out[i] = (int32_t)buf[i].index;
    qsort(out, (size_t)take, sizeof(int32_t), cmp_i32);
    for (int64_t i = take; i < k; ++i) out[i] = -1;
  }
  free(buf);
}

/* --------------------------------------------------------- core attention */

/*
 * Softmax attention of one query head over a list of rows, two passes in
 * double ([HA] section I, scaled dot-product attention; [HA] VI, key = value
 * = the compressed entries for MQA).  rows[e] indexes the row-major [*][c]
 * arrays k and v of dtype kv_dtype; q_h is the decoded query head.
 * o_h (double[c]) and *lse (natural log of the softmax denominator of the
 * scaled scores) are written; an empty list gives o = 0, lse = -inf (R7).
 */
static void attend_one(const double* q_h, int kv_dtype, const void* k, const void* v, int64_t kv_base,
                       const int64_t* rows, int64_t n_rows, int64_t c, double scale, double* sc, double* o_h,
                       double* lse) {
  for (int64_t d = 0; d < c; ++d) o_h[d] = 0.0;
  if (n_rows == 0) {
    *lse = -INFINITY;
    return;
  }
  double mx = -INFINITY;
  for (int64_t e = 0; e < n_rows; ++e) {
    double dot = 0.0;
    for (int64_t d = 0; d < c; ++d) dot += q_h[d] * load_elem(kv_dtype, k, (kv_base + rows[e]) * c + d);
    sc[e] = dot * scale;
    if (sc[e] > mx) mx = sc[e];
  }
  double den = 0.0;
  for (int64_t e = 0; e < n_rows; ++e) den += exp(sc[e] - mx);
  for (int64_t e = 0; e < n_rows; ++e) {
    double p = exp(sc[e] - mx) / den;
    for (int64_t d = 0; d < c; ++d) o_h[d] += p * load_elem(kv_dtype, v, (kv_base + rows[e]) * c + d);
  }
  *lse = mx + log(den);
}

static void decode_query_head(int dtype, const void* q, int64_t off, int64_t c, double* q_h) {
  for (int64_t d = 0; d < c; ++d) q_h[d] = load_elem(dtype, q, off + d);
}

/*
 * CSA core ([HA] V.3): every head of query (b, j) attends the entries listed
 * in idx[b][j][0..k) (entries < 0 are padding and skipped).
 * q [B][n_q][n_h][c]; kc, vc [B][N][c]; o [B][n_q][n_h][c]; lse [B][n_q][n_h].
 */
void orc_csa_attend(int dtype, const void* q, const void* kc, const void* vc, const int32_t* idx, int64_t B,
                    int64_t n_q, int64_t n_h, int64_t c, int64_t N, int64_t k, double scale, double* o,
                    double* lse) {
  int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(k > 0 ? k : 1));
  double* sc = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
  double* q_h = (double*)malloc(sizeof(double) * (size_t)c);
  for (int64_t b = 0; b < B; ++b)
    for (int64_t j = 0; j < n_q; ++j) {
      int64_t nr = 0;
      for (int64_t i = 0; i < k; ++i) {
        int32_t s = idx[(b * n_q + j) * k + i];
        if (s >= 0 && s < N) rows[nr++] = s;
      }
      for (int64_t h = 0; h < n_h; ++h) {
        int64_t qo = ((b * n_q + j) * n_h + h) * c;
        decode_query_head(dtype, q, qo, c, q_h);
        attend_one(q_h, dtype, kc, vc, b * N, rows, nr, c, scale, sc, &o[qo], &lse[(b * n_q + j) * n_h + h]);
      }
    }
  free(rows);
  free(sc);
  free(q_h);
}

/*
 * HCA core ([HA] VI, "dense over that tiny compressed set"): query (b, j) at
 * position t = q_pos0 + j attends every entry s < floor((t+1)/m') (R5).
 */
void orc_hca_attend(int dtype, const void* q, const void* kc, const void* vc, int64_t B, int64_t n_q,
                    int64_t n_h, int64_t c, int64_t N, int64_t m, int64_t q_pos0, double scale, double* o,
                    double* lse) {
  int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N > 0 ? N : 1));
  double* sc = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
  double* q_h = (double*)malloc(sizeof(double) * (size_t)c);
  for (int64_t s = 0; s < N; ++s) rows[s] = s;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t j = 0; j < n_q; ++j) {
      int64_t vis = orc_visible(q_pos0 + j, m);
      if (vis > N) vis = N;
      for (int64_t h = 0; h < n_h; ++h) {
        int64_t qo = ((b * n_q + j) * n_h + h) * c;
        decode_query_head(dtype, q, qo, c, q_h);
        attend_one(q_h, dtype, kc, vc, b * N, rows, vis, c, scale, sc, &o[qo], &lse[(b * n_q + j) * n_h + h]);
      }
    }
  free(rows);
  free(sc);
  free(q_h);
}

/*
 * Sliding-window branch and merge ([DV4] steps 4-5; [KE] section 9 "keep last
 * 128 exact").  Query (b, j) at t = q_pos0 + j attends the raw rows at
 * absolute positions max(0, t-n_win+1) .. t, held in kw/vw [B][n_kv][c] whose
 * row 0 is absolute position kv_pos0.  The result (o_w, lse_w) is merged with
 * the compressed branch (o_in, lse_in) as one softmax over the union (R8):
 *   L = logaddexp(lse_in, lse_w);  out = e^(lse_in-L) o_in + e^(lse_w-L) o_w.
 * o_in [B][n_q][n_h][c], lse_in [B][n_q][n_h] (double); out like o_in;
 * lse_out (optional, may be NULL) receives L.
 */
void orc_swa_merge(int dtype, const void* q, const void* kw, const void* vw, int64_t B, int64_t n_q, int64_t n_h,
                   int64_t c, int64_t n_kv, int64_t kv_pos0, int64_t q_pos0, int64_t n_win, double scale,
                   const double* o_in, const double* lse_in, double* out, double* lse_out) {
  int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n_win > 0 ? n_win : 1));
  double* sc = (double*)malloc(sizeof(double) * (size_t)(n_win > 0 ? n_win : 1));
  double* q_h = (double*)malloc(sizeof(double) * (size_t)c);
  double* o_w = (double*)malloc(sizeof(double) * (size_t)c);
  for (int64_t b = 0; b < B; ++b)
    for (int64_t j = 0; j < n_q; ++j) {
      int64_t t = q_pos0 + j;
      int64_t cnt = orc_window_count(t, n_win);
      int64_t nr = 0;
      for (int64_t u = t - cnt + 1; u <= t; ++u) rows[nr++] = u - kv_pos0;
      for (int64_t h = 0; h < n_h; ++h) {
        int64_t qo = ((b * n_q + j) * n_h + h) * c;
        int64_t li = (b * n_q + j) * n_h + h;
        double lse_w;
        decode_query_head(dtype, q, qo, c, q_h);
        attend_one(q_h, dtype, kw, vw, b * n_kv, rows, nr, c, scale, sc, o_w, &lse_w);
        double a = lse_in[li], bb = lse_w;
        double L;
        if (a == -INFINITY && bb == -INFINITY)
          L = -INFINITY;
        else {
          double mx = a > bb ? a : bb;
          L = mx + log(exp(a - mx) + exp(bb - mx));
        }
        for (int64_t d = 0; d < c; ++d) {
          double v = 0.0;
          if (L != -INFINITY) {
            if (a != -INFINITY) v += exp(a - L) * o_in[qo + d];
            if (bb != -INFINITY) v += exp(bb - L) * o_w[d];
          }
          out[qo + d] = v;
        }
        if (lse_out) lse_out[li] = L;
      }
    }
  free(rows);
  free(sc);
  free(q_h);
  free(o_w);
}

/* ------------------------------------------------- in-branch operations
 * [HA] section IV (the hybrid attention block): inside both branches the queries
 * and the compressed KV entries are RMS-normalised, only the last 64 dimensions
 * carry rotary position encoding, and every head has a learnable attention sink.
 * The pages name these without formulas; the textbook definitions are written
 * out below, with the rotary convention of [JH] "The Code: RoPE Helpers"
 * (consecutive dimension pairs, frequency theta^(-2i/d)).
 */

/* RMSNorm of each row: y[d] = x[d] / sqrt(mean_d x^2 + eps) * gamma[d].
 * x, y [rows][c] double; gamma [c] double (NULL = all ones). */
void orc_rmsnorm(const double* x, int64_t rows, int64_t c, const double* gamma, double eps, double* y) {
  for (int64_t r = 0; r < rows; ++r) {
    double ss = 0.0;
    for (int64_t d = 0; d < c; ++d) ss += x[r * c + d] * x[r * c + d];
    double inv = 1.0 / sqrt(ss / (double)c + eps);
    for (int64_t d = 0; d < c; ++d) y[r * c + d] = x[r * c + d] * inv * (gamma ? gamma[d] : 1.0);
  }
}

/* Partial rotary encoding: the last rope_dims dimensions of each row, taken as
 * consecutive pairs (2i, 2i+1) of that slice, are rotated by the angle
 * pos[r] * theta^(-2i / rope_dims); the first c - rope_dims dimensions are copied.
 * x, y [rows][c] double; pos [rows] (the row's position, any real value). */
void orc_rope_partial(const double* x, int64_t rows, int64_t c, int64_t rope_dims, const double* pos,
                      double theta, double* y) {
  int64_t d0 = c - rope_dims;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t d = 0; d < d0; ++d) y[r * c + d] = x[r * c + d];
    for (int64_t i = 0; i < rope_dims / 2; ++i) {
      double freq = pow(theta, -(double)(2 * i) / (double)rope_dims);
      double ang = pos[r] * freq;
      double re = x[r * c + d0 + 2 * i], im = x[r * c + d0 + 2 * i + 1];
      y[r * c + d0 + 2 * i] = re * cos(ang) - im * sin(ang);
      y[r * c + d0 + 2 * i + 1] = re * sin(ang) + im * cos(ang);
    }
  }
}

/* Attention sink: one more logit s_h per head in the softmax denominator, with no
 * value.  Given the branch's result (o, lse) over its attended multiset,
 *   out = o * exp(lse - L),   L = log(exp(lse) + exp(s_h)).
 * o, out [rows][n_h][c], lse, lse_out [rows][n_h] double; sink [n_h] double
 * (-inf = no sink).  lse_out may be NULL. */
void orc_sink_merge(const double* o, const double* lse, int64_t rows, int64_t n_h, int64_t c, const double* sink,
                    double* out, double* lse_out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t h = 0; h < n_h; ++h) {
      double a = lse[r * n_h + h], s = sink[h], L;
      if (a == -INFINITY && s == -INFINITY)
        L = -INFINITY;
      else {
        double mx = a > s ? a : s;
        L = mx + log(exp(a - mx) + exp(s - mx));
      }
      double w = (a == -INFINITY) ? 0.0 : exp(a - L);
      for (int64_t d = 0; d < c; ++d) out[(r * n_h + h) * c + d] = w * o[(r * n_h + h) * c + d];
      if (lse_out) lse_out[r * n_h + h] = L;
    }
}

/* ------------------------------------------------ grouped output projection
 * [HA] section V.3 ("Core attention and grouped output"): the concatenated head
 * outputs (n_h heads of c values) are split into g groups of n_h/g consecutive
 * heads; group j's (n_h/g)*c values are projected by its own d_g x (n_h/g)*c
 * matrix, and the g results are concatenated (g*d_g values per row).
 * o [rows][n_h*c], W [g][d_g][(n_h/g)*c], out [rows][g*d_g], all double.
 */
void orc_grouped_out_proj(const double* o, const double* W, int64_t rows, int64_t n_h, int64_t c, int64_t g,
                          int64_t d_g, double* out) {
  int64_t in_g = (n_h / g) * c;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t j = 0; j < g; ++j)
      for (int64_t e = 0; e < d_g; ++e) {
        double acc = 0.0;
        for (int64_t d = 0; d < in_g; ++d) acc += W[(j * d_g + e) * in_g + d] * o[r * n_h * c + j * in_g + d];
        out[r * g * d_g + j * d_g + e] = acc;
      }
}
