/*
 * CSA2 oracle: a plain, slow, single-threaded CPU definition of the CSA2
 * sparse-attention hot path, in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check
 * and the benchmark's CPU-baseline leg may load this code.  It shares no
 * code, header, table or helper with the CUDA library; the two meet only in
 * the seeded input bytes.
 *
 * Sources (web pages on DeepSeek-V4.1-Flash; citations name the page and its
 * section):
 *  [P2]  modelscope.csdn.net release summary, section "CSA2": three static
 *        layer modes Full / Reindex / Reuse that share main KV and indexer K
 *        and reuse top-k indices; FP4 main-KV cache in E2M1 with one E4M3
 *        scale per 16 channels.
 *  [P4a] wkq9411.github.io paper walkthrough, section 1.(4) "CSA2": a
 *        lightweight indexer scores main-KV entries with indexer Q and K and
 *        keeps the top-k entries per query; each query attends the selected
 *        entries; ratio-m compression without overlap.
 *  [P4b] same page, 1.(4).1 "Cross-Layer KV and Index Reuse": what each mode
 *        computes and what it takes from earlier layers.
 *  [P4c] same page, 1.(4).2 "Hierarchical Sparse Indexer": the first Full
 *        layer builds a candidate pool, later Reindex layers score only pool
 *        positions and take their own top-k there.
 *  [P4d] same page, 1.(5).4 "FP4 Main KV Cache": E2M1 values, one E4M3 scale
 *        per 16 channels, no second-level global scale, largest magnitude
 *        448 x 6 = 2688, quantised after RoPE, dequantised before attention.
 *  [P4e] same page, 3.(2).1 "Model settings": 64 main query heads of 512 dims.
 *  [P4f] same page, 1.(5).4: the indexer query and key are FP4 in the OCP
 *        MXFP4 format.
 *
 * Readings where the pages are silent:
 *  R1  scale byte = E4M3(absmax/6) rounded to nearest even, saturating at 448;
 *      code = E2M1 value nearest to the exact quotient |x|/scale, ties to the
 *      even code; sign bit = sign bit of x; scale 0 gives magnitude code 0.
 *  R2  row layout: D/2 code bytes (channel 2j in the low nibble of byte j),
 *      then D/16 scale bytes (byte b covers channels 16b..16b+15).
 *  R3  indexer score = sum over indexer heads of the dot product of that
 *      head's q with the entry's single (head-shared) indexer K vector.
 *  R4  entry j of a ratio-r context is visible to the query at token
 *      position pos iff r*j + r - 1 <= pos (the entry's last token is not
 *      in the future).  No position array means every entry is visible.
 *  R5  top-k = the min(k, visible) visible entries ranked by score
 *      descending then index ascending; returned in ascending index order,
 *      padded with -1.
 *  R6  hierarchical pool = the top-P of the Full layer's scores (flat pool of
 *      positions); a Reindex layer scores only pool entries and ranks them by
 *      (score desc, entry index asc).
 *  R7  attention: K = V = the dequantised 512-channel latent shared by all
 *      heads (MQA over the latent); logits = scale * <q_h, v_j>; softmax over
 *      the selected entries; -1 slots are skipped; no valid slot gives
 *      o = 0 and lse = -inf.  No RoPE is applied (the cache is quantised
 *      after RoPE).
 *  R8  a Reuse layer takes the indices of the nearest preceding Full or
 *      Reindex layer.
 *  R10 SWA branch [P4a], [P4d]: each layer's sliding-window KV holds one
 *      512-channel latent per token in plain E4M3 (the page keeps SWA KV in
 *      FP8; RMS-normalised latents stay far inside E4M3's +-448), kept per
 *      sequence in a ring of swa_ring rows (token t at row t mod swa_ring).
 *      The query at position pos attends tokens max(0, pos - n_win + 1) ..
 *      pos (its own token included) together with its selected entries, in
 *      one softmax; K = V = the decoded latent, same scale.
 *  R11 MXFP4 indexer [P4d] (indexer q and K in OCP MXFP4): per block of 32
 *      values, shared exponent = floor(log2(absmax)) - 2 (2 = the largest
 *      E2M1 exponent), clamped to the E8M0 range, scale 2^shared; elements
 *      E2M1 nearest to value / scale (an exact quotient), ties to the even
 *      code, saturating at 6; sign bit = sign of the value; an all-zero block
 *      takes scale byte 0.  Row: D/2 code bytes (element 2j in the low nibble
 *      of byte j) then D/32 scale bytes (E8M0, 2^(byte - 127)).
 *  R9  blockwise candidate pool [P4c]: entries are cut into aligned blocks of
 *      `block` consecutive entries; a block's score is the largest score of
 *      its visible entries (a block without one is no candidate); the
 *      n_blocks best blocks by (score desc, block index asc) are kept; the
 *      pool is the visible entries of the kept blocks in ascending order,
 *      padded with -1 to n_blocks * block slots.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* Formats [P2], [P4d]                                                     */
/* ---------------------------------------------------------------------- */

/* E2M1: sign bit, 2 exponent bits (bias 1), 1 mantissa bit.  Magnitudes of
 * codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_value(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double mag = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
  return s ? -mag : mag;
}

/* E4M3 (OCP 8-bit floating point, "e4m3fn"): sign, 4 exponent bits (bias 7),
 * 3 mantissa bits, no infinities, S.1111.111 is NaN. */
double orc_e4m3_value(int byte) {
  int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) mag = (m / 8.0) * ldexp(1.0, -6);
  else mag = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
  return s ? -mag : mag;
}

/* Nearest E4M3 byte to v, ties to the even mantissa (even byte), saturating
 * to the largest finite magnitude 448.  Exhaustive search over the 127
 * non-negative finite codes. */
int orc_e4m3_encode(double v) {
  if (isnan(v)) return 0x7F;
  int sign = signbit(v) ? 0x80 : 0;
  double a = fabs(v);
  if (a >= 448.0) return sign | 0x7E;
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    double d = fabs(orc_e4m3_value(c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return sign | best;
}

/* Nearest of the 8 E2M1 magnitudes to q >= 0, ties to the even code. */
int orc_e2m1_encode_magnitude(double q) {
  int best = 0;
  double best_d = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double d = fabs(orc_e2m1_value(c) - q);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return best;
}

static double bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* ---------------------------------------------------------------------- */
/* FP4 main-KV quantise / dequantise [P4d], readings R1, R2                */
/* ---------------------------------------------------------------------- */

int64_t orc_fp4_row_bytes(int d) { return d / 2 + d / 16; }

/* x: fp32 [n_rows][d] -> out: [n_rows][d/2 + d/16] bytes.  d % 16 == 0. */
void orc_quantize_kv_fp4(const float* x, int64_t n_rows, int d, uint8_t* out) {
  int64_t rb = orc_fp4_row_bytes(d);
  for (int64_t r = 0; r < n_rows; ++r) {
    const float* xr = x + r * d;
    uint8_t* codes = out + r * rb;
    uint8_t* scales = codes + d / 2;
    memset(codes, 0, (size_t)(d / 2));
    for (int b = 0; b < d / 16; ++b) {
      double amax = 0.0;
      for (int i = 0; i < 16; ++i) amax = fmax(amax, fabs((double)xr[16 * b + i]));
      /* amax/6 and |x|/s below are fp64 quotients of an fp32 value by a
       * number of at most 4 significant bits.  Such a quotient can equal a
       * rounding midpoint (at most 5 significant bits) only if the exact
       * quotient equals it, because an fp32 dividend next to 6 x midpoint
       * (resp. s x midpoint) differs from it by at least 2^-24 relative,
       * far above fp64's 2^-53; so rounding the fp64 quotient is rounding
       * the exact quotient. */
      int sbyte = orc_e4m3_encode(amax / 6.0);
      double s = orc_e4m3_value(sbyte);
      scales[b] = (uint8_t)sbyte;
      for (int i = 0; i < 16; ++i) {
        int ch = 16 * b + i;
        double xv = (double)xr[ch];
        int mag = (s == 0.0) ? 0 : orc_e2m1_encode_magnitude(fabs(xv) / s);
        int code = (signbit(xv) ? 8 : 0) | mag;
        codes[ch / 2] |= (uint8_t)((ch & 1) ? (code << 4) : code);
      }
    }
  }
}

/* One row of [d/2 + d/16] bytes -> d values: code value x scale. */
void orc_dequantize_row(const uint8_t* row, int d, double* out) {
  const uint8_t* scales = row + d / 2;
  for (int ch = 0; ch < d; ++ch) {
    int code = (ch & 1) ? (row[ch / 2] >> 4) : (row[ch / 2] & 15);
    out[ch] = orc_e2m1_value(code) * orc_e4m3_value(scales[ch / 16]);
  }
}

/* ---------------------------------------------------------------------- */
/* MXFP4 indexer rows [P4f], reading R11                                   */
/* ---------------------------------------------------------------------- */

/* E8M0 (OCP MX shared scale): 2^(byte - 127); 0xFF (NaN) is never written. */
double orc_e8m0_value(int byte) { return ldexp(1.0, byte - 127); }

int64_t orc_mxfp4_row_bytes(int d) { return d / 2 + d / 32; }

/* x: fp32 [n_rows][d] -> out: [n_rows][d/2 + d/32].  d % 32 == 0. */
void orc_quantize_mxfp4(const float* x, int64_t n_rows, int d, uint8_t* out) {
  int64_t rb = orc_mxfp4_row_bytes(d);
  for (int64_t r = 0; r < n_rows; ++r) {
    const float* xr = x + r * d;
    uint8_t* codes = out + r * rb;
    uint8_t* scales = codes + d / 2;
    memset(codes, 0, (size_t)(d / 2));
    for (int b = 0; b < d / 32; ++b) {
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs((double)xr[32 * b + i]));
      int shared = -127;
      if (amax > 0.0) {
        int e;
        frexp(amax, &e);           /* amax = m 2^e, m in [0.5, 1): floor(log2 amax) = e - 1 */
        shared = (e - 1) - 2;
        if (shared < -127) shared = -127;
        if (shared > 127) shared = 127;
      }
      scales[b] = (uint8_t)(shared + 127);
      double X = ldexp(1.0, shared);
      for (int i = 0; i < 32; ++i) {
        int ch = 32 * b + i;
        double xv = (double)xr[ch];
        int mag = orc_e2m1_encode_magnitude(fabs(xv) / X); /* exact: X is a power of two */
        int code = (signbit(xv) ? 8 : 0) | mag;
        codes[ch / 2] |= (uint8_t)((ch & 1) ? (code << 4) : code);
      }
    }
  }
}

void orc_dequantize_mxfp4_row(const uint8_t* row, int d, double* out) {
  const uint8_t* scales = row + d / 2;
  for (int ch = 0; ch < d; ++ch) {
    int code = (ch & 1) ? (row[ch / 2] >> 4) : (row[ch / 2] & 15);
    out[ch] = orc_e2m1_value(code) * orc_e8m0_value(scales[ch / 32]);
  }
}

void orc_dequantize_kv_fp4(const uint8_t* rows, int64_t n_rows, int d, double* out) {
  int64_t rb = orc_fp4_row_bytes(d);
  for (int64_t r = 0; r < n_rows; ++r) orc_dequantize_row(rows + r * rb, d, out + r * d);
}

/* ---------------------------------------------------------------------- */
/* Causal visibility [P4a], reading R4                                     */
/* ---------------------------------------------------------------------- */

int64_t orc_n_visible(const int32_t* q_pos, int q, int ratio, int64_t N) {
  if (!q_pos) return N;
  /* visibility is monotone in j, so the visible entries form a prefix;
   * count it straight from the definition */
  int64_t pos = q_pos[q], n = 0;
  while (n < N && (int64_t)ratio * n + ratio - 1 <= pos) ++n;
  return n;
}

/* ---------------------------------------------------------------------- */
/* Indexer scores [P4a], [P4b], reading R3                                 */
/* ---------------------------------------------------------------------- */

/* scores[q][j] = sum_h sum_d qI[q][h][d] * KI[seq(q)][j][d] for visible j,
 * -inf otherwise.  q_fp8 [B][H_I][D_I], k_fp8 [S][N][D_I] (sequence s at
 * offset s * kv_seq_stride entries), scores [B][N]. */
/* Indexer rows: fmt 0 = E4M3 [D_I] bytes, fmt 1 = MXFP4 (R11). */
static int64_t idx_row_bytes(int D_I, int fmt) {
  return fmt ? orc_mxfp4_row_bytes(D_I) : D_I;
}
static void idx_row_values(const uint8_t* row, int D_I, int fmt, double* out) {
  if (fmt) {
    orc_dequantize_mxfp4_row(row, D_I, out);
  } else {
    for (int d = 0; d < D_I; ++d) out[d] = orc_e4m3_value(row[d]);
  }
}

void orc_index_scores_fmt(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I, int D_I,
                          int64_t N, int64_t kv_seq_stride, int q_per_seq, const int32_t* q_pos,
                          int ratio, int fmt, double* scores) {
  int64_t rb = idx_row_bytes(D_I, fmt);
  double* kj = (double*)malloc(sizeof(double) * D_I);
  double* qv = (double*)malloc(sizeof(double) * H_I * D_I);
  for (int q = 0; q < B; ++q) {
    const uint8_t* kseq = k_fp8 + (int64_t)(q / q_per_seq) * kv_seq_stride * rb;
    int64_t nv = orc_n_visible(q_pos, q, ratio, N);
    for (int h = 0; h < H_I; ++h)
      idx_row_values(q_fp8 + ((int64_t)q * H_I + h) * rb, D_I, fmt, qv + (int64_t)h * D_I);
    for (int64_t j = 0; j < N; ++j) {
      if (j >= nv) {
        scores[(int64_t)q * N + j] = -INFINITY;
        continue;
      }
      idx_row_values(kseq + j * rb, D_I, fmt, kj);
      double s = 0.0;
      for (int h = 0; h < H_I; ++h) {
        double dot = 0.0;
        for (int d = 0; d < D_I; ++d) dot += qv[h * D_I + d] * kj[d];
        s += dot;
      }
      scores[(int64_t)q * N + j] = s;
    }
  }
  free(kj);
  free(qv);
}

void orc_index_scores(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I, int D_I,
                      int64_t N, int64_t kv_seq_stride, int q_per_seq, const int32_t* q_pos,
                      int ratio, double* scores) {
  orc_index_scores_fmt(q_fp8, k_fp8, B, H_I, D_I, N, kv_seq_stride, q_per_seq, q_pos, ratio, 0,
                       scores);
}

/* ---------------------------------------------------------------------- */
/* Top-k [P4a], reading R5                                                 */
/* ---------------------------------------------------------------------- */

typedef struct {
  double s;
  int64_t j;
} cand_t;

static int cmp_rank(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* Rank n candidates, write the first min(k, n) entry ids in ascending order
 * to out[0..k), pad with -1. */
static void select_topk(cand_t* c, int64_t n, int k, int32_t* out) {
  qsort(c, (size_t)n, sizeof(cand_t), cmp_rank);
  int64_t take = n < k ? n : k;
  for (int64_t t = 0; t < take; ++t) out[t] = (int32_t)c[t].j;
  qsort(out, (size_t)take, sizeof(int32_t), cmp_i32);
  for (int64_t t = take; t < k; ++t) out[t] = -1;
}

/* scores [B][N] -> idx [B][k]; only visible entries (R4) are candidates. */
void orc_topk(const double* scores, int B, int64_t N, int k, const int32_t* q_pos, int ratio,
              int32_t* idx) {
  cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (N > 0 ? N : 1));
  for (int q = 0; q < B; ++q) {
    int64_t nv = orc_n_visible(q_pos, q, ratio, N);
    for (int64_t j = 0; j < nv; ++j) {
      c[j].s = scores[(int64_t)q * N + j];
      c[j].j = j;
    }
    select_topk(c, nv, k, idx + (int64_t)q * k);
  }
  free(c);
}

/* ---------------------------------------------------------------------- */
/* Hierarchical Sparse Indexer, blockwise candidate pool [P4c], reading R9 */
/* ---------------------------------------------------------------------- */

/* scores [B][N] -> pool [B][n_blocks * block].  The steps follow the page:
 * block score = max of the index scores in the block, the top-scoring
 * blocks are chosen, and the positions they cover form the pool. */
void orc_block_pool(const double* scores, int B, int64_t N, const int32_t* q_pos, int ratio,
                    int block, int n_blocks, int32_t* pool) {
  int64_t nb_max = (N + block - 1) / block;
  cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (nb_max > 0 ? nb_max : 1));
  int32_t* chosen = (int32_t*)malloc(sizeof(int32_t) * (n_blocks > 0 ? n_blocks : 1));
  int64_t P = (int64_t)n_blocks * block;
  for (int q = 0; q < B; ++q) {
    int64_t nv = orc_n_visible(q_pos, q, ratio, N);
    int64_t nb = (nv + block - 1) / block; /* blocks holding a visible entry */
    for (int64_t b = 0; b < nb; ++b) {
      double m = -INFINITY;
      for (int64_t j = b * block; j < (b + 1) * block && j < nv; ++j)
        if (scores[(int64_t)q * N + j] > m) m = scores[(int64_t)q * N + j];
      c[b].s = m;
      c[b].j = b;
    }
    select_topk(c, nb, n_blocks, chosen); /* chosen blocks, ascending, -1 padded */
    int64_t o = 0;
    for (int t = 0; t < n_blocks; ++t) {
      if (chosen[t] < 0) continue;
      for (int64_t j = (int64_t)chosen[t] * block; j < ((int64_t)chosen[t] + 1) * block && j < nv; ++j)
        pool[(int64_t)q * P + o++] = (int32_t)j;
    }
    for (; o < P; ++o) pool[(int64_t)q * P + o] = -1;
  }
  free(c);
  free(chosen);
}

/* ---------------------------------------------------------------------- */
/* Hierarchical Sparse Indexer, Reindex-in-pool [P4c], reading R6          */
/* ---------------------------------------------------------------------- */

/* For each query, score only the entries listed in pool[q][0..P) (-1 slots
 * skipped) and keep the top-k of them by (score desc, entry id asc). */
void orc_hier_pool_index_fmt(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I, int D_I,
                             int64_t N, int64_t kv_seq_stride, int q_per_seq, const int32_t* pool,
                             int P, int k, int fmt, int32_t* idx) {
  int64_t rb = idx_row_bytes(D_I, fmt);
  cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (P > 0 ? P : 1));
  double* qv = (double*)malloc(sizeof(double) * H_I * D_I);
  double* kj = (double*)malloc(sizeof(double) * D_I);
  for (int q = 0; q < B; ++q) {
    const uint8_t* kseq = k_fp8 + (int64_t)(q / q_per_seq) * kv_seq_stride * rb;
    for (int h = 0; h < H_I; ++h)
      idx_row_values(q_fp8 + ((int64_t)q * H_I + h) * rb, D_I, fmt, qv + (int64_t)h * D_I);
    int64_t n = 0;
    for (int p = 0; p < P; ++p) {
      int32_t j = pool[(int64_t)q * P + p];
      if (j < 0 || j >= N) continue;
      idx_row_values(kseq + (int64_t)j * rb, D_I, fmt, kj);
      double s = 0.0;
      for (int h = 0; h < H_I; ++h) {
        double dot = 0.0;
        for (int d = 0; d < D_I; ++d) dot += qv[h * D_I + d] * kj[d];
        s += dot;
      }
      c[n].s = s;
      c[n].j = j;
      ++n;
    }
    select_topk(c, n, k, idx + (int64_t)q * k);
  }
  free(c);
  free(qv);
  free(kj);
}

void orc_hier_pool_index(const uint8_t* q_fp8, const uint8_t* k_fp8, int B, int H_I, int D_I,
                         int64_t N, int64_t kv_seq_stride, int q_per_seq, const int32_t* pool,
                         int P, int k, int32_t* idx) {
  orc_hier_pool_index_fmt(q_fp8, k_fp8, B, H_I, D_I, N, kv_seq_stride, q_per_seq, pool, P, k, 0,
                          idx);
}

/* ---------------------------------------------------------------------- */
/* Sparse MQA attention over the selected FP4 entries [P4a], [P4d], R7     */
/* ---------------------------------------------------------------------- */

/* Attention of one query's heads over n gathered latent rows v [n][D]. */
static void attend(const uint16_t* q_bf16, int H, int D, const double* v, int n, double scale,
                   double* out, double* lse, double* logit, double* qh) {
  for (int h = 0; h < H; ++h) {
    double* o = out + (int64_t)h * D;
    for (int c = 0; c < D; ++c) qh[c] = bf16_value(q_bf16[(int64_t)h * D + c]);
    if (n == 0) {
      for (int c = 0; c < D; ++c) o[c] = 0.0;
      if (lse) lse[h] = -INFINITY;
      continue;
    }
    double m = -INFINITY;
    for (int t = 0; t < n; ++t) {
      double dot = 0.0;
      for (int c = 0; c < D; ++c) dot += qh[c] * v[(int64_t)t * D + c];
      logit[t] = scale * dot;
      if (logit[t] > m) m = logit[t];
    }
    double l = 0.0;
    for (int t = 0; t < n; ++t) {
      logit[t] = exp(logit[t] - m); /* now the unnormalised weight */
      l += logit[t];
    }
    for (int c = 0; c < D; ++c) o[c] = 0.0;
    for (int t = 0; t < n; ++t) {
      double p = logit[t] / l;
      for (int c = 0; c < D; ++c) o[c] += p * v[(int64_t)t * D + c];
    }
    if (lse) lse[h] = m + log(l);
  }
}

/* q_bf16 [B][H][D] (bf16 bits), kv_fp4 [S][N][D/2 + D/16], idx [B][k]
 * -> out [B][H][D] (fp64), lse [B][H] (fp64, may be NULL).
 * With swa_kv (R10): E4M3 [S][swa_ring][D]; the window of n_win tokens
 * ending at q_pos[q] joins the selected entries in the same softmax
 * (swa_kv NULL or n_win 0: no window). */
void orc_sparse_attn_swa(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H, int D,
                         int64_t N, int64_t kv_seq_stride, int q_per_seq, const int32_t* idx,
                         int k, const uint8_t* swa_kv, int64_t swa_ring, int n_win,
                         const int32_t* q_pos, double scale, double* out, double* lse) {
  int64_t rb = orc_fp4_row_bytes(D);
  int64_t cap = (int64_t)(k > 0 ? k : 0) + (swa_kv && n_win > 0 ? n_win : 0);
  double* v = (double*)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1) * D);
  double* logit = (double*)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1));
  double* qh = (double*)malloc(sizeof(double) * D);
  for (int q = 0; q < B; ++q) {
    int64_t s = q / q_per_seq;
    const uint8_t* kvseq = kv_fp4 + s * kv_seq_stride * rb;
    /* gather and dequantise the selected rows */
    int n = 0;
    for (int t = 0; t < k; ++t) {
      int32_t j = idx[(int64_t)q * k + t];
      if (j < 0 || j >= N) continue;
      orc_dequantize_row(kvseq + (int64_t)j * rb, D, v + (int64_t)n * D);
      ++n;
    }
    /* the query's own sliding window of the layer's SWA KV */
    if (swa_kv && n_win > 0 && q_pos && q_pos[q] >= 0) {
      int64_t pos = q_pos[q];
      int64_t t0 = pos - n_win + 1 > 0 ? pos - n_win + 1 : 0;
      for (int64_t t = t0; t <= pos; ++t) {
        const uint8_t* row = swa_kv + (s * swa_ring + t % swa_ring) * D;
        for (int c = 0; c < D; ++c) v[(int64_t)n * D + c] = orc_e4m3_value(row[c]);
        ++n;
      }
    }
    attend(q_bf16 + (int64_t)q * H * D, H, D, v, n, scale, out + (int64_t)q * H * D,
           lse ? lse + (int64_t)q * H : NULL, logit, qh);
  }
  free(v);
  free(logit);
  free(qh);
}

void orc_sparse_attn(const uint16_t* q_bf16, const uint8_t* kv_fp4, int B, int H, int D, int64_t N,
                     int64_t kv_seq_stride, int q_per_seq, const int32_t* idx, int k,
                     double scale, double* out, double* lse) {
  orc_sparse_attn_swa(q_bf16, kv_fp4, B, H, D, N, kv_seq_stride, q_per_seq, idx, k, NULL, 0, 0,
                      NULL, scale, out, lse);
}

/* ---------------------------------------------------------------------- */
/* Layer modes Full / Reindex / Reuse [P4b], [P4c], reading R8             */
/* ---------------------------------------------------------------------- */

enum { ORC_FULL = 0, ORC_REINDEX = 1, ORC_REUSE = 2 };

/* Runs n_layers layers over one shared FP4 main KV and indexer K.
 *   modes[l]          FULL / REINDEX / REUSE; layer 0 must be FULL
 *   q_bf16[l]         [B][H][D] main query of layer l
 *   qi_fp8[l]         [B][H_I][D_I] indexer query (ignored for REUSE)
 *   out[l], lse[l]    [B][H][D], [B][H] outputs (lse may be NULL)
 *   idx_out[l]        [B][k] indices layer l attended (written for every layer)
 *   indexer_fmt       0: indexer q / K in E4M3 [D_I]; 1: in MXFP4 rows (R11)
 *   swa_kv[l]         E4M3 [S][swa_ring][D] SWA KV of layer l (R10), or NULL;
 *                     with n_win > 0 each layer also attends its window
 *   pool_out          [B][pool_size] when pool_size > 0 (built by FULL layers):
 *                     pool_block == 0: the top pool_size entries (R6);
 *                     pool_block > 0: the blockwise pool of pool_size /
 *                     pool_block blocks of pool_block entries (R9)
 * Returns 0, or -1 for an invalid schedule. */
int orc_layer_group(int n_layers, const int* modes, const uint16_t* const* q_bf16,
                    const uint8_t* const* qi_fp8, double* const* out, double* const* lse,
                    int32_t* const* idx_out, const uint8_t* kv_fp4, const uint8_t* ki_fp8, int B,
                    int H, int H_I, int D, int D_I, int64_t N, int64_t kv_seq_stride,
                    int q_per_seq, const int32_t* q_pos, int ratio, int k, int pool_size,
                    int pool_block, int32_t* pool_out, const uint8_t* const* swa_kv,
                    int64_t swa_ring, int n_win, int indexer_fmt, double scale) {
  if (n_layers < 1 || modes[0] != ORC_FULL) return -1;
  if (pool_block < 0 || (pool_block > 0 && pool_size % pool_block != 0)) return -1;
  double* scores = (double*)malloc(sizeof(double) * (size_t)B * (size_t)(N > 0 ? N : 1));
  const int32_t* latest = NULL;
  for (int l = 0; l < n_layers; ++l) {
    int32_t* idx = idx_out[l];
    if (modes[l] == ORC_FULL) {
      orc_index_scores_fmt(qi_fp8[l], ki_fp8, B, H_I, D_I, N, kv_seq_stride, q_per_seq, q_pos,
                           ratio, indexer_fmt, scores);
      orc_topk(scores, B, N, k, q_pos, ratio, idx);
      if (pool_size > 0 && pool_block == 0)
        orc_topk(scores, B, N, pool_size, q_pos, ratio, pool_out);
      else if (pool_size > 0)
        orc_block_pool(scores, B, N, q_pos, ratio, pool_block, pool_size / pool_block, pool_out);
      latest = idx;
    } else if (modes[l] == ORC_REINDEX) {
      if (pool_size > 0) {
        orc_hier_pool_index_fmt(qi_fp8[l], ki_fp8, B, H_I, D_I, N, kv_seq_stride, q_per_seq,
                                pool_out, pool_size, k, indexer_fmt, idx);
      } else {
        orc_index_scores_fmt(qi_fp8[l], ki_fp8, B, H_I, D_I, N, kv_seq_stride, q_per_seq, q_pos,
                             ratio, indexer_fmt, scores);
        orc_topk(scores, B, N, k, q_pos, ratio, idx);
      }
      latest = idx;
    } else if (modes[l] == ORC_REUSE) {
      memcpy(idx, latest, sizeof(int32_t) * (size_t)B * (size_t)k);
    } else {
      free(scores);
      return -1;
    }
    orc_sparse_attn_swa(q_bf16[l], kv_fp4, B, H, D, N, kv_seq_stride, q_per_seq, idx, k,
                        swa_kv ? swa_kv[l] : NULL, swa_ring, n_win, q_pos, scale, out[l],
                        lse ? lse[l] : NULL);
  }
  free(scores);
  return 0;
}
