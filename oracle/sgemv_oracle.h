/*
 * sgemv_oracle.h -- CPU oracle for the N:4 "2bit-CSR" INT4 SparseGemv.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this code: only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code with the CUDA library.
 *
 * Source of the method: Dong et al., "Efficient LLM ad generation via model
 * compression and parallel verification" (arXiv 2605.11582).
 *   - N:M pruning, 2:4 for critical layers and 1:4 for the others:
 *     section 3.2, "Sparsification", and the Figure 1 caption.
 *   - the importance criterion, Eq. (3); with a constant activation norm and
 *     a zero gradient term it orders weights by |W_ij| (magnitude pruning).
 *   - group-wise quantization FP16 -> INT4 with per-layer group size:
 *     section 1 ("Our core idea") and section 3.2, "Adaptive group quantization".
 *   - the index-compressed 2bit-CSR format: section 1, contribution 1.
 *   - the INT4 weight-only mixed-sparsity GEMV: section 1, contribution 2,
 *     and section 3.3 (truncated in the source text).
 * The pages leave the byte layout, the rounding rules and the zero-point
 * convention open; the readings taken here are listed with each function.
 *
 * Canonical layout (one row r of an R x K weight, P = K*N/4 kept weights):
 *   vals[r][j/2]  : INT4 code of kept weight j, low nibble for even j.
 *                   Row stride ceil(P/2) bytes.
 *   idx [r][j/4]  : 2-bit in-quad position of kept weight j at bits 2*(j%4).
 *                   Row stride ceil(P/4) bytes.  Kept weight j lies in quad
 *                   floor(j/N); positions within a quad ascend.
 *   scale[r][G], zero[r][G] : IEEE binary16 bit patterns, G = 0..K/g-1.
 * Dequantised weight: W_hat[r][4*floor(j/N) + pos_j] = (q_j - zero) * scale.
 *
 * Parity status: every function below is pinned by the CPU test suite
 * (brute force, invariants, closed forms, library routines); the paper's own
 * byte layout and quantiser are not printed on the pages, so the readings
 * above are this project's, not the paper's.
 */
#ifndef SGEMV_ORACLE_H
#define SGEMV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Error codes returned by the oracle (0 = success). */
#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_NONFINITE (-6)
#define ORC_ERR_RANGE (-7)

/* IEEE-754 binary16 conversions, round to nearest, ties to even. */
uint16_t orc_f64_to_f16(double v);
uint16_t orc_f32_to_f16(float v);
double orc_f16_to_f64(uint16_t h);

/* Canonical byte counts of one row. */
int64_t orc_vals_row_bytes(int64_t cols, int n_keep);
int64_t orc_idx_row_bytes(int64_t cols, int n_keep);

/* O1: magnitude N:4 pruning.  pos is rows x (cols/4) x n_keep, ascending
 * within a quad.  Returns ORC_ERR_NONFINITE on NaN/Inf anywhere in W. */
int orc_prune(const float* W, int64_t rows, int64_t cols, int n_keep,
              uint8_t* pos);

/* O2: asymmetric INT4 quantisation per (row, group of `group` dense
 * columns) of the kept weights.  q is rows x P codes in 0..15.
 * Returns ORC_ERR_RANGE if a scale does not fit binary16. */
int orc_quantize(const float* W, const uint8_t* pos, int64_t rows,
                 int64_t cols, int n_keep, int group, uint8_t* q,
                 uint16_t* scale, uint16_t* zero);

/* O3: encode (pos, q) into the canonical vals / idx bytes. */
void orc_encode(const uint8_t* pos, const uint8_t* q, int64_t rows,
                int64_t cols, int n_keep, uint8_t* vals, uint8_t* idx);

/* Inverse of O3. */
void orc_decode(const uint8_t* vals, const uint8_t* idx, int64_t rows,
                int64_t cols, int n_keep, uint8_t* pos, uint8_t* q);

/* O1 by the paper's Eq. 3 importance score
 *   score = |W_ij| * xnorm[j] + |W_ij| * |grad_ij|
 * in binary32 as written (two products, one sum, each rounded once), the N
 * largest per quad, ties to the lower column.  xnorm: cols finite values
 * >= 0; grad: rows x cols or NULL (zero gradient). */
int orc_prune_scored(const float* W, const float* xnorm, const float* grad,
                     int64_t rows, int64_t cols, int n_keep, uint8_t* pos);

/* orc_prune_scored + O2 + O3. */
int orc_pack_scored(const float* W, const float* xnorm, const float* grad,
                    int64_t rows, int64_t cols, int n_keep, int group,
                    uint8_t* vals, uint8_t* idx, uint16_t* scale,
                    uint16_t* zero);

/* O1 + O2 + O3 in one call, scratch allocated internally. */
int orc_pack(const float* W, int64_t rows, int64_t cols, int n_keep,
             int group, uint8_t* vals, uint8_t* idx, uint16_t* scale,
             uint16_t* zero);

/* O4: dense fp64 dequantised rows [row0, row0+nrows) into out
 * (nrows x cols, row-major). */
void orc_dequant_rows(const uint8_t* vals, const uint8_t* idx,
                      const uint16_t* scale, const uint16_t* zero,
                      int64_t cols, int n_keep, int group, int64_t row0,
                      int64_t nrows, double* out);

/* O5: y[i][mm] = sum_c W_hat[rows_list[i]][c] * x[mm][c] in fp64, naive
 * loops in ascending c.  x is m x cols binary16 bit patterns.  y is
 * n_list x m (one line per listed row). */
void orc_matvec(const uint8_t* vals, const uint8_t* idx,
                const uint16_t* scale, const uint16_t* zero, int64_t cols,
                int n_keep, int group, const uint16_t* x, int m,
                const int64_t* rows_list, int64_t n_list, double* y);

/* Per-row group sizes: row r uses group row_group[r] (a divisor of cols);
 * scale/zero hold each row's cols / row_group[r] entries after those of
 * the rows before it.  Each row is exactly the single-row case of the
 * uniform-group functions above. */
int orc_quantize_rowg(const float* W, const uint8_t* pos, int64_t rows,
                      int64_t cols, int n_keep, const int* row_group,
                      uint8_t* q, uint16_t* scale, uint16_t* zero);
int orc_pack_rowg(const float* W, int64_t rows, int64_t cols, int n_keep,
                  const int* row_group, uint8_t* vals, uint8_t* idx,
                  uint16_t* scale, uint16_t* zero);
void orc_dequant_rows_rowg(const uint8_t* vals, const uint8_t* idx,
                           const uint16_t* scale, const uint16_t* zero,
                           int64_t cols, int n_keep, const int* row_group,
                           int64_t row0, int64_t nrows, double* out);
void orc_matvec_rowg(const uint8_t* vals, const uint8_t* idx,
                     const uint16_t* scale, const uint16_t* zero, int64_t rows,
                     int64_t cols, int n_keep, const int* row_group,
                     const uint16_t* x, int m, const int64_t* rows_list,
                     int64_t n_list, double* y);

#ifdef __cplusplus
}
#endif

#endif /* SGEMV_ORACLE_H */
