/*
 * Plain-C twin of the CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A second, independently written float64 implementation of the In-Place TTT
 * fast-weight SwiGLU layer, used by the tests on tiny inputs to cross-check
 * oracle/oracle.py.  It is written with explicit loops only (no BLAS) and shares
 * no code with the Python oracle or with the CUDA library.
 *
 * Definitions followed (zhichai.net "In-Place TTT：给LLM装上"临时记忆插槽"，
 * 让它边读边学"):
 *   §3.1 gated MLP:     Z = SiLU(H W_gate^T) * (H W_up^T)
 *   §3.3 target:        V = CausalConv1D(X0) W_target  (depthwise, zero left pad k-1)
 *   §3.2 chunk loop:    O_i = Z_i W^T with the current W, then
 *   §3.3 update rule:   W <- W + eta V_i^T Z_i
 * Layouts (row-major): H, X0 [T,d]; W_gate, W_up [f,d]; W_down0 [d,f];
 * W_target [d,d] (right-multiplied); conv_w [d,k]; O [T,d]; W_final [d,f].
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

int twin_sequence_forward(const double *H, const double *X0, const double *W_gate,
                          const double *W_up, const double *W_down0, const double *W_target,
                          const double *conv_w, long T, long d, long f, long C, long k,
                          double eta, double *O, double *W_final) {
  if (T < 0 || d <= 0 || f <= 0 || C <= 0 || k <= 0) return 1;
  double *Z = (double *)calloc((size_t)(T > 0 ? T : 1) * (size_t)f, sizeof(double));
  double *Y = (double *)calloc((size_t)(T > 0 ? T : 1) * (size_t)d, sizeof(double));
  double *V = (double *)calloc((size_t)(T > 0 ? T : 1) * (size_t)d, sizeof(double));
  double *W = (double *)malloc((size_t)d * (size_t)f * sizeof(double));
  if (!Z || !Y || !V || !W) {
    free(Z); free(Y); free(V); free(W);
    return 2;
  }
  /* gated MLP, one output element at a time */
  for (long t = 0; t < T; ++t) {
    for (long j = 0; j < f; ++j) {
      double a = 0.0, u = 0.0;
      for (long c = 0; c < d; ++c) {
        a += H[t * d + c] * W_gate[j * d + c];
        u += H[t * d + c] * W_up[j * d + c];
      }
      double sig = 1.0 / (1.0 + exp(-a));
      Z[t * f + j] = a * sig * u;
    }
  }
  /* causal depthwise convolution: output t sees X0[t-k+1 .. t] */
  for (long t = 0; t < T; ++t) {
    for (long c = 0; c < d; ++c) {
      double acc = 0.0;
      for (long s = 0; s < k; ++s) {
        long src = t - (k - 1) + s;
        if (src >= 0) acc += conv_w[c * k + s] * X0[src * d + c];
      }
      Y[t * d + c] = acc;
    }
  }
  /* target projection, W_target right-multiplied */
  for (long t = 0; t < T; ++t) {
    for (long o = 0; o < d; ++o) {
      double acc = 0.0;
      for (long c = 0; c < d; ++c) acc += Y[t * d + c] * W_target[c * d + o];
      V[t * d + o] = acc;
    }
  }
  memcpy(W, W_down0, (size_t)d * (size_t)f * sizeof(double));
  for (long lo = 0; lo < T; lo += C) {
    long hi = lo + C < T ? lo + C : T;
    /* output of the chunk with the weight left by the earlier chunks */
    for (long t = lo; t < hi; ++t) {
      for (long o = 0; o < d; ++o) {
        double acc = 0.0;
        for (long j = 0; j < f; ++j) acc += Z[t * f + j] * W[o * f + j];
        O[t * d + o] = acc;
      }
    }
    /* one step after the chunk */
    for (long o = 0; o < d; ++o) {
      for (long j = 0; j < f; ++j) {
        double acc = 0.0;
        for (long t = lo; t < hi; ++t) acc += V[t * d + o] * Z[t * f + j];
        W[o * f + j] += eta * acc;
      }
    }
  }
  memcpy(W_final, W, (size_t)d * (size_t)f * sizeof(double));
  free(Z); free(Y); free(V); free(W);
  return 0;
}
