/*
 * Second CPU oracle for the AWQ GEMM-layout linear, in plain C.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests load it (and the build step compiles it); the CUDA
 * library and its binding never link, load or call it, and it includes nothing from them.
 * It is written separately from the numpy oracle (awq_oracle.py) so that the two can be
 * checked against each other: they share no code, only the definitions below.
 *
 * Definitions followed:
 *  - Unpack (tensref.org/formats/awq, "Reader"): nibble i (bits 4i .. 4i+3) of the 32-bit
 *    word c of a row holds output column 8c + ORDER[i], ORDER = {0, 2, 4, 6, 1, 3, 5, 7};
 *    zeros are packed the same way.  Words are taken as their unsigned bit pattern.
 *  - 8-bit codes (GPTQModel wiki "AWQ", "Saved formats and packing": widths other than 4
 *    form a plain little-endian bit stream): byte i of word c holds column 4c + i.
 *  - Dequantize (format page, "Reader"; reject rule AWQ-005: no +1 on the zero): for input
 *    row k the group row is g = k / G (G = K when group_size is -1), and
 *    w = (code - zero) * scale, evaluated in fp32 (exact: a 9-bit integer times an 11-bit
 *    significand).
 *  - Linear: y[m][n] = sum over k = 0, 1, ..., K-1 of x[m][k] * w[k][n], in fp64, plus
 *    bias[n] when a bias is given (format page: "bias ... optional, shape [out_features]").
 *  - fp16 inputs are widened by decoding the IEEE 754 binary16 fields directly.
 *
 * Every entry point returns 0, or 1 when the shape is invalid.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

static const int ORDER[8] = {0, 2, 4, 6, 1, 3, 5, 7};

/* IEEE 754 binary16: sign bit 15, exponent bits 10-14 (bias 15), fraction bits 0-9. */
static float half_to_float(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1F;
  const int f = h & 0x3FF;
  float v;
  if (e == 0)
    v = ldexpf((float)f, -24); /* subnormal: f * 2^-24 */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexpf((float)(1024 + f), e - 25); /* (1 + f / 2^10) * 2^(e - 15) */
  return sign ? -v : v;
}

void awq_oracle_widen_f16(const uint16_t* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = half_to_float(in[i]);
}

static int resolve_group(int64_t K, int64_t group_size, int64_t* G) {
  *G = group_size == -1 ? K : group_size;
  return (K > 0 && *G > 0 && K % *G == 0) ? 0 : 1;
}

/* w [K][N] fp32 from bits-wide codes (4 or 8). */
int awq_oracle_dequant_f32(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                           int64_t K, int64_t N, int64_t group_size, int bits, float* w) {
  int64_t G;
  if (resolve_group(K, group_size, &G)) return 1;
  if (bits != 4 && bits != 8) return 1;
  const int per_word = 32 / bits;
  if (N <= 0 || N % per_word != 0) return 1;
  const int64_t C = N / per_word;
  for (int64_t k = 0; k < K; ++k) {
    const int64_t g = k / G;
    for (int64_t c = 0; c < C; ++c) {
      const uint32_t q = (uint32_t)qweight[k * C + c];
      const uint32_t z = (uint32_t)qzeros[g * C + c];
      for (int i = 0; i < per_word; ++i) {
        int64_t n;
        uint32_t code, zero;
        if (bits == 4) {
          n = 8 * c + ORDER[i];
          code = (q >> (4 * i)) & 0xFu;
          zero = (z >> (4 * i)) & 0xFu;
        } else {
          n = 4 * c + i;
          code = (q >> (8 * i)) & 0xFFu;
          zero = (z >> (8 * i)) & 0xFFu;
        }
        w[k * N + n] = ((float)code - (float)zero) * half_to_float(scales[g * N + n]);
      }
    }
  }
  return 0;
}

/* y [M][N] fp64.  Each output sums its K products in increasing k; rows of y are
 * independent, so they are shared out over threads without changing any sum. */
int awq_oracle_gemm_f64(const uint16_t* x, const int32_t* qweight, const int32_t* qzeros,
                        const uint16_t* scales, const uint16_t* bias, int64_t M, int64_t K,
                        int64_t N, int64_t group_size, int bits, double* y) {
  if (M < 0) return 1;
  float* w = (float*)malloc((size_t)(K > 0 ? K : 1) * (size_t)(N > 0 ? N : 1) * sizeof(float));
  if (!w) return 1;
  if (awq_oracle_dequant_f32(qweight, qzeros, scales, K, N, group_size, bits, w)) {
    free(w);
    return 1;
  }
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    double* row = y + m * N;
    for (int64_t n = 0; n < N; ++n) row[n] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double xk = (double)half_to_float(x[m * K + k]);
      const float* wk = w + k * N;
      for (int64_t n = 0; n < N; ++n) row[n] += xk * (double)wk[n];
    }
    if (bias)
      for (int64_t n = 0; n < N; ++n) row[n] += (double)half_to_float(bias[n]);
  }
  free(w);
  return 0;
}
