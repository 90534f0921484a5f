/*
 * Slow, plain fp64 CPU oracle for the packed-batch forward of a Mamba2
 * mixer's varlen conv + selective state-space scan under continuous batching.
 * TEST INFRASTRUCTURE ONLY: nothing on the product path may include, link or
 * call this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code with the CUDA path.
 *
 * What it follows:
 *  - "Continuous batching: model support tracker": Mamba2 mixers keep a conv
 *    state and an SSM state per request, and the groundwork the page asks for
 *    is a varlen scan with per-sequence states, like the varlen causal
 *    convolution; "Continuous batching for linear attention layers": those
 *    states sit in one block per request, read from the zeroed trash block
 *    while the request has no past and overwritten in place.
 *  - The Mamba2 scan (Dao and Gu, "Transformers are SSMs: Generalized Models
 *    and Efficient Algorithms Through Structured State Space Duality", 2024,
 *    the SSD recurrence with a scalar-times-identity A per head):
 *        dt_t = softplus(dt_raw_t + dt_bias),   a_t = exp(-exp(A_log) dt_t),
 *        h_t  = a_t h_{t-1} + dt_t x_t B_t^T,   y_t = h_t C_t + D x_t,
 *    per head, with h the P x N state (P = head dim, N = state size); heads
 *    of one group share B and C (head h reads group h / (H/G)).
 *
 * The conv is the same varlen causal depthwise conv1d + SiLU as the gated
 * delta net oracle (oracle_conv_silu_seq, gdn_oracle.c), over the channels
 * x | B | C (H*P + 2*G*N of them).  Token by token, no chunking or
 * reordering; fp64 logical arrays.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

void oracle_conv_silu_seq(int L, int C, int K, const double* x, const double* tail,
                          const double* w, int ch0, int nch, double* y);
void oracle_conv_tail_update(int L, int C, int K, const double* x, const double* old_tail,
                             double* new_tail);

static double ssd_softplus(double x) {
  if (x > 0.0) return x + log1p(exp(-x));
  return log1p(exp(x));
}

/*
 * The scan of ONE (sequence, head) chain, given its conv outputs.
 *   x : [L][P]  the head's x channels      B, C : [L][N]  its group's B and C
 *   dt: [L]     raw dt (dt_bias added here)
 *   h : [P][N]  state, in: h_0, out: h_L   y : [L][P]
 */
void oracle_ssd_scan_head(int L, int P, int N, const double* x, const double* B, const double* C,
                          const double* dt, double A_log, double dt_bias, double Dskip,
                          double* h, double* y) {
  for (int t = 0; t < L; ++t) {
    const double* xt = x + (size_t)t * P;
    const double* Bt = B + (size_t)t * N;
    const double* Ct = C + (size_t)t * N;
    double d = ssd_softplus(dt[t] + dt_bias);
    double a = exp(-exp(A_log) * d);
    for (int p = 0; p < P; ++p) {
      double acc = 0.0;
      for (int n = 0; n < N; ++n) {
        double v = a * h[(size_t)p * N + n] + d * xt[p] * Bt[n];
        h[(size_t)p * N + n] = v;
        acc += v * Ct[n];
      }
      y[(size_t)t * P + p] = acc + Dskip * xt[p];
    }
  }
}

/*
 * Whole packed forward, on logical fp64 arrays.
 *   xbc      : [T][Cc] with Cc = H*P + 2*G*N, channels x | B | C
 *   dt       : [T][H]
 *   cu, blk, has_past, skip: as the gated delta net oracle
 *   w        : [Cc][K]; A_log, dt_bias, Dskip: [H]
 *   conv_st  : [num_blocks][K-1][Cc] in/out
 *   ssm_st   : [num_blocks][H][P][N] in/out
 *   y        : [T][H][P]; rows of skipped sequences are left untouched
 * Returns the number of OpenMP threads used.
 */
int oracle_ssd_forward(int T, int Nseq, int H, int P, int N, int G, int K, int num_blocks,
                       const double* xbc, const double* dt, const int32_t* cu, const int32_t* blk,
                       const uint8_t* has_past, const uint8_t* skip, const double* w,
                       const double* A_log, const double* dt_bias, const double* Dskip,
                       double* conv_st, double* ssm_st, double* y, int nthreads) {
  (void)T;
  (void)num_blocks;
  const int Cc = H * P + 2 * G * N;
  const int W = K - 1;
  const int ratio = H / G;
  const size_t conv_blk = (size_t)W * Cc;
  const size_t ssm_head = (size_t)P * N;
  const size_t ssm_blk = (size_t)H * ssm_head;
  int used = 1;

  /* Phase 1: every (sequence, head) chain reads its source block. */
  int npairs = Nseq * H;
  double** hfin = (double**)calloc((size_t)npairs, sizeof(double*));
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
  {
#pragma omp single
    used = omp_get_num_threads();
  }
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int pair = 0; pair < npairs; ++pair) {
    int s = pair / H, hd = pair % H;
    int L = cu[s + 1] - cu[s];
    if (blk[s] < 0 || L <= 0 || (skip && skip[s])) continue;
    int src = has_past[s] ? blk[s] : 0;
    int g = hd / ratio;
    const double* xs = xbc + (size_t)cu[s] * Cc;
    const double* tail = conv_st + (size_t)src * conv_blk;
    double* xy = (double*)malloc(sizeof(double) * (size_t)L * P);
    double* By = (double*)malloc(sizeof(double) * (size_t)L * N);
    double* Cy = (double*)malloc(sizeof(double) * (size_t)L * N);
    double* dts = (double*)malloc(sizeof(double) * (size_t)L);
    double* yo = (double*)malloc(sizeof(double) * (size_t)L * P);
    double* h = (double*)malloc(sizeof(double) * ssm_head);
    oracle_conv_silu_seq(L, Cc, K, xs, tail, w, hd * P, P, xy);
    oracle_conv_silu_seq(L, Cc, K, xs, tail, w, H * P + g * N, N, By);
    oracle_conv_silu_seq(L, Cc, K, xs, tail, w, H * P + G * N + g * N, N, Cy);
    for (int t = 0; t < L; ++t) dts[t] = dt[(size_t)(cu[s] + t) * H + hd];
    memcpy(h, ssm_st + (size_t)src * ssm_blk + (size_t)hd * ssm_head, sizeof(double) * ssm_head);
    oracle_ssd_scan_head(L, P, N, xy, By, Cy, dts, A_log[hd], dt_bias[hd], Dskip[hd], h, yo);
    for (int t = 0; t < L; ++t)
      memcpy(y + ((size_t)(cu[s] + t) * H + hd) * P, yo + (size_t)t * P, sizeof(double) * P);
    hfin[pair] = h;
    free(xy); free(By); free(Cy); free(dts); free(yo);
  }

  /* Phase 2: new conv tails from the source blocks, before any overwrite. */
  double** tails = (double**)calloc((size_t)Nseq, sizeof(double*));
  for (int s = 0; s < Nseq; ++s) {
    int L = cu[s + 1] - cu[s];
    if (blk[s] < 0 || L <= 0 || (skip && skip[s])) continue;
    int src = has_past[s] ? blk[s] : 0;
    tails[s] = (double*)malloc(sizeof(double) * conv_blk);
    oracle_conv_tail_update(L, Cc, K, xbc + (size_t)cu[s] * Cc, conv_st + (size_t)src * conv_blk,
                            tails[s]);
  }

  /* Phase 3: overwrite each request's block in place. */
  for (int s = 0; s < Nseq; ++s) {
    if (!tails[s]) continue;
    memcpy(conv_st + (size_t)blk[s] * conv_blk, tails[s], sizeof(double) * conv_blk);
    free(tails[s]);
    for (int hd = 0; hd < H; ++hd) {
      double* h = hfin[s * H + hd];
      memcpy(ssm_st + (size_t)blk[s] * ssm_blk + (size_t)hd * ssm_head, h, sizeof(double) * ssm_head);
      free(h);
    }
  }
  free(tails);
  free(hfin);
  return used;
}
