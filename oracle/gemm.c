/*
 * gemm.c -- oracle for the consumer of the block-scaled FP8 tiles: a GEMM
 * whose FP8 partial sums are promoted to FP32 scaling every 128 elements of
 * K.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h).
 *
 * [P1] "Loss scaling, FP8, and the failure that never crashes", section
 * "FP8 needs a finer-grained fix than a single scale factor": FP8 tensor
 * cores accumulate in a narrow register, so DeepSeek-V3's kernels promote
 * partial sums to FP32 at short intervals; [P5] "Mixed precision and FP8
 * training", section "FP8 training": the partial sum is promoted to FP32
 * every 128 elements (DeepGEMM), activations carry 1x128 and weights
 * 128x128 scales.  With A = [M, K] codes and 1x128 scales sa[M, K/128], and
 * B = [N, K] codes (the weight, rows are output features) with 128x128
 * scales sb[N/128, K/128]:
 *   D[m][n] = sum over K-blocks kb of
 *             sa[m][kb] * sb[n/128][kb] * sum_{k in kb} dec(A[m][k]) * dec(B[n][k]).
 * A and B may be in different formats ([P5] "FP8 training": E4M3 for the
 * forward tensors, E5M2 for gradients, so a backward GEMM multiplies E5M2
 * gradients by E4M3 weights): dec() is each operand's own decoding.
 * Computed here in double: every FP8 product is exact, and a block of 128
 * of them is summed exactly (their magnitudes span less than 2^53); the
 * scaling and the sum over blocks round in double only.
 */
#include <stdint.h>

#include "oracle.h"

double orc_gemm_fp8_block_elem(const uint8_t* qa, const float* sa, const uint8_t* qb,
                               const float* sb, int64_t K, int64_t m, int64_t n, int fmt_a,
                               int fmt_b) {
  const int64_t nkb = K / 128;
  double acc = 0.0;
  for (int64_t kb = 0; kb < nkb; ++kb) {
    double p = 0.0;
    for (int64_t k = kb * 128; k < (kb + 1) * 128; ++k)
      p += orc_fp8_decode(qa[m * K + k], fmt_a) * orc_fp8_decode(qb[n * K + k], fmt_b);
    acc += p * (double)sa[m * nkb + kb] * (double)sb[(n / 128) * nkb + kb];
  }
  return acc;
}

void orc_gemm_fp8_block(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                        int64_t M, int64_t N, int64_t K, int fmt_a, int fmt_b, double* d) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      d[m * N + n] = orc_gemm_fp8_block_elem(qa, sa, qb, sb, K, m, n, fmt_a, fmt_b);
}
