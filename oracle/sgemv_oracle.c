/*
 * sgemv_oracle.c -- plain, slow, obviously correct CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY (see sgemv_oracle.h): used by the test suite,
 * the smoke check and the benchmark's CPU-baseline leg, never by the
 * product path.  Compiled with -O2 -ffp-contract=off and without
 * -ffast-math, so every float operation below is one correctly rounded
 * IEEE operation in the order written.
 *
 * Method source: Dong et al., "Efficient LLM ad generation via model
 * compression and parallel verification" (arXiv 2605.11582), sections
 * 1 (contributions 1-3), 3.2 (adaptive group quantization; sparsification;
 * Eq. 3) and 3.3.  Readings of what those sections leave open:
 *   R1 pruning order: keep the N kept weights of largest |w| in each quad
 *      of 4 along K; on equal |w| the lower column wins; +0 and -0 are
 *      equal.  (Eq. 3 with equal activation norms and no gradient term.)
 *   R2 quantiser: asymmetric, w_hat = (q - z) * s with q, z integers in
 *      [0, 15]; the range [lo, hi] always includes 0; s is (hi - lo) / 15
 *      rounded to binary16; rounding is round-half-to-even throughout.
 *   R3 layout: the canonical 2bit-CSR bytes described in the header.
 *   R11 importance score: Eq. 3 evaluated in binary32 as written (see
 *      orc_prune_scored); magnitude pruning (R1) is its case of equal norms
 *      and zero gradient.
 */
#include "sgemv_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* IEEE-754 binary16 (1 sign bit, 5 exponent bits with bias 15, 10
 * fraction bits).  Normal numbers: (1024 + f) * 2^(e - 25) for biased
 * exponent e in 1..30; subnormals: f * 2^-24.                          */
/* ------------------------------------------------------------------ */

double orc_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int f = h & 0x3FF;
  double v;
  if (e == 31) {
    v = f ? NAN : INFINITY;
  } else if (e == 0) {
    v = ldexp((double)f, -24);
  } else {
    v = ldexp((double)(1024 + f), e - 25);
  }
  return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even.  A binary64 value
 * is sig * 2^(E - 52) with a 53-bit integer significand sig.  The binary16
 * unit in the last place at that magnitude is 2^(max(E, -14) - 10); the
 * result is the count of those units, rounded, placed in the bit pattern. */
uint16_t orc_f64_to_f16(double v) {
  uint64_t b;
  memcpy(&b, &v, sizeof b);
  uint16_t sign = (uint16_t)((b >> 48) & 0x8000u);
  int be = (int)((b >> 52) & 0x7FF);
  uint64_t frac = b & ((1ULL << 52) - 1);
  if (be == 0x7FF) return (uint16_t)(sign | (frac ? 0x7E00u : 0x7C00u));
  if (be == 0) return sign; /* zero or binary64 subnormal: far below 2^-25 */
  int E = be - 1023;
  if (E > 15) return (uint16_t)(sign | 0x7C00u); /* >= 2^16: overflow */
  uint64_t sig = (1ULL << 52) | frac;
  int unit_exp = (E < -14 ? -14 : E) - 10;
  int shift = 52 - (E - unit_exp); /* bits of sig below one unit */
  if (shift > 53) return sign;     /* value < 2^-25 * ...: below half a unit */
  uint64_t units = sig >> shift;
  uint64_t rem = sig & ((1ULL << shift) - 1);
  uint64_t half = 1ULL << (shift - 1);
  if (rem > half || (rem == half && (units & 1))) units++;
  uint64_t bits;
  if (E < -14) {
    bits = units; /* subnormal; units == 1024 is the smallest normal */
  } else {
    bits = ((uint64_t)(E + 14) << 10) + units; /* units in [1024, 2048] */
  }
  if (bits >= 0x7C00u) bits = 0x7C00u;
  return (uint16_t)(sign | bits);
}

uint16_t orc_f32_to_f16(float v) {
  /* float -> double is exact, so this is a single rounding. */
  return orc_f64_to_f16((double)v);
}

/* ------------------------------------------------------------------ */

int64_t orc_vals_row_bytes(int64_t cols, int n_keep) {
  int64_t p = cols / 4 * n_keep;
  return (p + 1) / 2;
}

int64_t orc_idx_row_bytes(int64_t cols, int n_keep) {
  int64_t p = cols / 4 * n_keep;
  return (p + 3) / 4;
}

static int shape_ok(int64_t rows, int64_t cols, int n_keep) {
  return rows >= 0 && cols >= 0 && cols % 4 == 0 &&
         (n_keep == 1 || n_keep == 2);
}

/* O1 (reading R1).  For each quad, element i is kept iff fewer than N
 * elements of the quad precede it in the order "larger |w| first, lower
 * column first on ties".  Kept positions are written in ascending order. */
int orc_prune(const float* W, int64_t rows, int64_t cols, int n_keep,
              uint8_t* pos) {
  if (!shape_ok(rows, cols, n_keep)) return ORC_ERR_ARG;
  int64_t quads = cols / 4;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t t = 0; t < quads; ++t) {
      const float* w = W + r * cols + 4 * t;
      float a[4];
      for (int i = 0; i < 4; ++i) {
        if (!isfinite(w[i])) return ORC_ERR_NONFINITE;
        a[i] = fabsf(w[i]);
      }
      uint8_t* out = pos + (r * quads + t) * n_keep;
      int k = 0;
      for (int i = 0; i < 4; ++i) {
        int ahead = 0;
        for (int j = 0; j < 4; ++j) {
          if (j == i) continue;
          if (a[j] > a[i] || (a[j] == a[i] && j < i)) ahead++;
        }
        if (ahead < n_keep) out[k++] = (uint8_t)i;
      }
    }
  }
  return ORC_OK;
}

/* O2 (reading R2), per (row r, group G of `group` dense columns), over the
 * group's kept values S, in fp32 with one rounding per operation:
 *   lo = min(0, min S), hi = max(0, max S)
 *   hi == lo:  s = 1.0, z = 0
 *   otherwise: s = f16_rne((hi - lo) / 15); s == 0 -> s = 2^-24
 *              z = clamp(rint(-lo / s), 0, 15)
 *   q = clamp(rint(w / s) + z, 0, 15)
 * A scale that rounds to binary16 infinity is a range error. */
int orc_quantize(const float* W, const uint8_t* pos, int64_t rows,
                 int64_t cols, int n_keep, int group, uint8_t* q,
                 uint16_t* scale, uint16_t* zero) {
  if (!shape_ok(rows, cols, n_keep)) return ORC_ERR_ARG;
  if (group <= 0 || group % 4 != 0 || cols % group != 0) return ORC_ERR_ARG;
  int64_t quads = cols / 4;
  int64_t P = quads * n_keep;
  int64_t ngroups = cols / group;
  int64_t qpg = group / 4; /* quads per group */
  for (int64_t r = 0; r < rows; ++r) {
    const float* wr = W + r * cols;
    for (int64_t G = 0; G < ngroups; ++G) {
      float lo = 0.0f, hi = 0.0f;
      for (int64_t t = G * qpg; t < (G + 1) * qpg; ++t) {
        for (int n = 0; n < n_keep; ++n) {
          float v = wr[4 * t + pos[(r * quads + t) * n_keep + n]];
          if (!isfinite(v)) return ORC_ERR_NONFINITE;
          if (v < lo) lo = v;
          if (v > hi) hi = v;
        }
      }
      uint16_t s16;
      int z;
      if (hi == lo) {
        s16 = 0x3C00u; /* 1.0 */
        z = 0;
      } else {
        float range = hi - lo;
        if (!isfinite(range)) return ORC_ERR_RANGE;
        float s32 = range / 15.0f;
        s16 = orc_f32_to_f16(s32);
        if ((s16 & 0x7FFFu) == 0x7C00u) return ORC_ERR_RANGE;
        if (s16 == 0) s16 = 0x0001u; /* smallest subnormal, 2^-24 */
        float sf = (float)orc_f16_to_f64(s16);
        float zf = rintf(-lo / sf);
        if (zf < 0.0f) zf = 0.0f;
        if (zf > 15.0f) zf = 15.0f;
        z = (int)zf;
      }
      float sf = (float)orc_f16_to_f64(s16);
      scale[r * ngroups + G] = s16;
      zero[r * ngroups + G] = orc_f32_to_f16((float)z);
      for (int64_t t = G * qpg; t < (G + 1) * qpg; ++t) {
        for (int n = 0; n < n_keep; ++n) {
          int64_t j = t * n_keep + n;
          float v = wr[4 * t + pos[(r * quads + t) * n_keep + n]];
          float qf = rintf(v / sf) + (float)z;
          if (qf < 0.0f) qf = 0.0f;
          if (qf > 15.0f) qf = 15.0f;
          q[r * P + j] = (uint8_t)qf;
        }
      }
    }
  }
  return ORC_OK;
}

/* O3 (reading R3). */
void orc_encode(const uint8_t* pos, const uint8_t* q, int64_t rows,
                int64_t cols, int n_keep, uint8_t* vals, uint8_t* idx) {
  int64_t P = cols / 4 * n_keep;
  int64_t vb = orc_vals_row_bytes(cols, n_keep);
  int64_t ib = orc_idx_row_bytes(cols, n_keep);
  memset(vals, 0, (size_t)(rows * vb));
  memset(idx, 0, (size_t)(rows * ib));
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t j = 0; j < P; ++j) {
      uint8_t code = q[r * P + j] & 0xF;
      uint8_t p = pos[r * P + j] & 0x3;
      vals[r * vb + j / 2] |= (uint8_t)(code << (4 * (j % 2)));
      idx[r * ib + j / 4] |= (uint8_t)(p << (2 * (j % 4)));
    }
  }
}

void orc_decode(const uint8_t* vals, const uint8_t* idx, int64_t rows,
                int64_t cols, int n_keep, uint8_t* pos, uint8_t* q) {
  int64_t P = cols / 4 * n_keep;
  int64_t vb = orc_vals_row_bytes(cols, n_keep);
  int64_t ib = orc_idx_row_bytes(cols, n_keep);
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t j = 0; j < P; ++j) {
      q[r * P + j] = (vals[r * vb + j / 2] >> (4 * (j % 2))) & 0xF;
      pos[r * P + j] = (idx[r * ib + j / 4] >> (2 * (j % 4))) & 0x3;
    }
  }
}

/* O1 with the paper's importance score (section 3.2, Eq. 3):
 *   score_ij = |W_ij| * ||X_j||_2 + |W_ij| * |dE/dW_ij|,
 * with the activation norms of the input columns and the loss gradient
 * supplied by the caller (grad NULL: zero gradient).  Reading R11: the
 * score is evaluated in binary32 exactly as written -- t1 = |w| * xn,
 * t2 = |w| * |g|, score = t1 + t2, each one rounding -- and each quad keeps
 * the N largest scores, the lower column first on equal scores, like R1.
 * NaN/Inf in W, xnorm or grad -> ORC_ERR_NONFINITE; a negative norm ->
 * ORC_ERR_ARG. */
int orc_prune_scored(const float* W, const float* xnorm, const float* grad,
                     int64_t rows, int64_t cols, int n_keep, uint8_t* pos) {
  if (!shape_ok(rows, cols, n_keep) || !xnorm) return ORC_ERR_ARG;
  for (int64_t c = 0; c < cols; ++c) {
    if (!isfinite(xnorm[c])) return ORC_ERR_NONFINITE;
    if (xnorm[c] < 0.0f) return ORC_ERR_ARG;
  }
  int64_t quads = cols / 4;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t t = 0; t < quads; ++t) {
      float sc[4];
      for (int i = 0; i < 4; ++i) {
        int64_t c = 4 * t + i;
        float w = W[r * cols + c];
        float g = grad ? grad[r * cols + c] : 0.0f;
        if (!isfinite(w) || !isfinite(g)) return ORC_ERR_NONFINITE;
        float aw = fabsf(w);
        float t1 = aw * xnorm[c];
        float t2 = aw * fabsf(g);
        sc[i] = t1 + t2;
      }
      uint8_t* out = pos + (r * quads + t) * n_keep;
      int k = 0;
      for (int i = 0; i < 4; ++i) {
        int ahead = 0;
        for (int j = 0; j < 4; ++j) {
          if (j == i) continue;
          if (sc[j] > sc[i] || (sc[j] == sc[i] && j < i)) ahead++;
        }
        if (ahead < n_keep) out[k++] = (uint8_t)i;
      }
    }
  }
  return ORC_OK;
}

/* O1 (by `pos` already chosen) + O2 + O3. */
static int pack_from_pos(const float* W, uint8_t* pos, int64_t rows,
                         int64_t cols, int n_keep, int group, uint8_t* vals,
                         uint8_t* idx, uint16_t* scale, uint16_t* zero) {
  int64_t P = cols / 4 * n_keep;
  size_t n = (size_t)(rows * P);
  uint8_t* q = (uint8_t*)malloc(n ? n : 1);
  if (!q) return ORC_ERR_ARG;
  int rc = orc_quantize(W, pos, rows, cols, n_keep, group, q, scale, zero);
  if (rc == ORC_OK) orc_encode(pos, q, rows, cols, n_keep, vals, idx);
  free(q);
  return rc;
}

int orc_pack_scored(const float* W, const float* xnorm, const float* grad,
                    int64_t rows, int64_t cols, int n_keep, int group,
                    uint8_t* vals, uint8_t* idx, uint16_t* scale,
                    uint16_t* zero) {
  if (!shape_ok(rows, cols, n_keep)) return ORC_ERR_ARG;
  int64_t P = cols / 4 * n_keep;
  size_t n = (size_t)(rows * P);
  uint8_t* pos = (uint8_t*)malloc(n ? n : 1);
  if (!pos) return ORC_ERR_ARG;
  int rc = orc_prune_scored(W, xnorm, grad, rows, cols, n_keep, pos);
  if (rc == ORC_OK)
    rc = pack_from_pos(W, pos, rows, cols, n_keep, group, vals, idx, scale, zero);
  free(pos);
  return rc;
}

int orc_pack(const float* W, int64_t rows, int64_t cols, int n_keep,
             int group, uint8_t* vals, uint8_t* idx, uint16_t* scale,
             uint16_t* zero) {
  if (!shape_ok(rows, cols, n_keep)) return ORC_ERR_ARG;
  int64_t P = cols / 4 * n_keep;
  size_t n = (size_t)(rows * P);
  uint8_t* pos = (uint8_t*)malloc(n ? n : 1);
  uint8_t* q = (uint8_t*)malloc(n ? n : 1);
  int rc = ORC_ERR_ARG;
  if (pos && q) {
    rc = orc_prune(W, rows, cols, n_keep, pos);
    if (rc == ORC_OK)
      rc = orc_quantize(W, pos, rows, cols, n_keep, group, q, scale, zero);
    if (rc == ORC_OK) orc_encode(pos, q, rows, cols, n_keep, vals, idx);
  }
  free(pos);
  free(q);
  return rc;
}

/* O4: scatter each kept weight's exact value (q - z) * s into its column. */
void orc_dequant_rows(const uint8_t* vals, const uint8_t* idx,
                      const uint16_t* scale, const uint16_t* zero,
                      int64_t cols, int n_keep, int group, int64_t row0,
                      int64_t nrows, double* out) {
  int64_t P = cols / 4 * n_keep;
  int64_t vb = orc_vals_row_bytes(cols, n_keep);
  int64_t ib = orc_idx_row_bytes(cols, n_keep);
  int64_t ngroups = group > 0 ? cols / group : 0;
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t r = row0 + i;
    double* o = out + i * cols;
    for (int64_t c = 0; c < cols; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < P; ++j) {
      int qj = (vals[r * vb + j / 2] >> (4 * (j % 2))) & 0xF;
      int pj = (idx[r * ib + j / 4] >> (2 * (j % 4))) & 0x3;
      int64_t c = 4 * (j / n_keep) + pj;
      int64_t G = c / group;
      double s = orc_f16_to_f64(scale[r * ngroups + G]);
      double z = orc_f16_to_f64(zero[r * ngroups + G]);
      o[c] = ((double)qj - z) * s;
    }
  }
}

/* O5: naive fp64 matvec over the dense dequantised row. */
void orc_matvec(const uint8_t* vals, const uint8_t* idx,
                const uint16_t* scale, const uint16_t* zero, int64_t cols,
                int n_keep, int group, const uint16_t* x, int m,
                const int64_t* rows_list, int64_t n_list, double* y) {
  double* row = (double*)malloc((size_t)(cols > 0 ? cols : 1) * sizeof(double));
  double* xd = (double*)malloc((size_t)(m * cols > 0 ? m * cols : 1) * sizeof(double));
  if (!row || !xd) {
    free(row);
    free(xd);
    for (int64_t i = 0; i < n_list * m; ++i) y[i] = NAN;
    return;
  }
  for (int64_t i = 0; i < (int64_t)m * cols; ++i) xd[i] = orc_f16_to_f64(x[i]);
  for (int64_t i = 0; i < n_list; ++i) {
    orc_dequant_rows(vals, idx, scale, zero, cols, n_keep, group,
                     rows_list[i], 1, row);
    for (int mm = 0; mm < m; ++mm) {
      const double* xm = xd + (int64_t)mm * cols;
      double acc = 0.0;
      for (int64_t c = 0; c < cols; ++c) acc += row[c] * xm[c];
      y[i * m + mm] = acc;
    }
  }
  free(row);
  free(xd);
}

/* ------------------------------------------------------------------ */
/* Per-row group sizes (the paper's finer groups for sensitive channels,
 * section 3.2 "Adaptive group quantization"): row r is quantised with its
 * own group size row_group[r]; its scale/zero entries follow those of the
 * rows before it (offset sum_{r' < r} cols / row_group[r']).  Every row is
 * the single-row case of the functions above.                          */
/* ------------------------------------------------------------------ */

static int row_groups_ok(const int* row_group, int64_t rows, int64_t cols) {
  if (!row_group) return 0;
  for (int64_t r = 0; r < rows; ++r) {
    int g = row_group[r];
    if (g <= 0 || cols % g != 0) return 0;
  }
  return 1;
}

int orc_quantize_rowg(const float* W, const uint8_t* pos, int64_t rows,
                      int64_t cols, int n_keep, const int* row_group,
                      uint8_t* q, uint16_t* scale, uint16_t* zero) {
  if (!shape_ok(rows, cols, n_keep) || !row_groups_ok(row_group, rows, cols))
    return ORC_ERR_ARG;
  int64_t P = cols / 4 * n_keep, off = 0;
  for (int64_t r = 0; r < rows; ++r) {
    int rc = orc_quantize(W + r * cols, pos + r * P, 1, cols, n_keep,
                          row_group[r], q + r * P, scale + off, zero + off);
    if (rc != ORC_OK) return rc;
    off += cols / row_group[r];
  }
  return ORC_OK;
}

int orc_pack_rowg(const float* W, int64_t rows, int64_t cols, int n_keep,
                  const int* row_group, uint8_t* vals, uint8_t* idx,
                  uint16_t* scale, uint16_t* zero) {
  if (!shape_ok(rows, cols, n_keep) || !row_groups_ok(row_group, rows, cols))
    return ORC_ERR_ARG;
  int64_t vb = orc_vals_row_bytes(cols, n_keep), ib = orc_idx_row_bytes(cols, n_keep);
  int64_t off = 0;
  for (int64_t r = 0; r < rows; ++r) {
    int rc = orc_pack(W + r * cols, 1, cols, n_keep, row_group[r], vals + r * vb,
                      idx + r * ib, scale + off, zero + off);
    if (rc != ORC_OK) return rc;
    off += cols / row_group[r];
  }
  return ORC_OK;
}

void orc_dequant_rows_rowg(const uint8_t* vals, const uint8_t* idx,
                           const uint16_t* scale, const uint16_t* zero,
                           int64_t cols, int n_keep, const int* row_group,
                           int64_t row0, int64_t nrows, double* out) {
  int64_t vb = orc_vals_row_bytes(cols, n_keep), ib = orc_idx_row_bytes(cols, n_keep);
  int64_t off = 0;
  for (int64_t r = 0; r < row0; ++r) off += cols / row_group[r];
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t r = row0 + i;
    orc_dequant_rows(vals + r * vb, idx + r * ib, scale + off, zero + off, cols,
                     n_keep, row_group[r], 0, 1, out + i * cols);
    off += cols / row_group[r];
  }
}

void orc_matvec_rowg(const uint8_t* vals, const uint8_t* idx,
                     const uint16_t* scale, const uint16_t* zero, int64_t rows,
                     int64_t cols, int n_keep, const int* row_group,
                     const uint16_t* x, int m, const int64_t* rows_list,
                     int64_t n_list, double* y) {
  int64_t vb = orc_vals_row_bytes(cols, n_keep), ib = orc_idx_row_bytes(cols, n_keep);
  int64_t* off = (int64_t*)malloc((size_t)(rows + 1) * sizeof(int64_t));
  if (!off) return;
  off[0] = 0;
  for (int64_t r = 0; r < rows; ++r) off[r + 1] = off[r] + cols / row_group[r];
  const int64_t zero_row = 0;
  for (int64_t i = 0; i < n_list; ++i) {
    int64_t r = rows_list[i];
    orc_matvec(vals + r * vb, idx + r * ib, scale + off[r], zero + off[r], cols,
               n_keep, row_group[r], x, m, &zero_row, 1, y + i * m);
  }
  free(off);
}
