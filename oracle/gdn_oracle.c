/*
 * Slow, plain fp64 CPU oracle for the packed-batch forward of a gated delta
 * net layer under continuous batching.  TEST INFRASTRUCTURE ONLY: nothing on
 * the product path may include, link or call this file; only the tests, the
 * smoke check and the benchmark's CPU-baseline leg use it.  It shares no code
 * with the CUDA path.
 *
 * What it follows:
 *  - "Continuous batching for linear attention layers" (PR description): a
 *    linear attention layer keeps, per request, the last inputs of its causal
 *    convolution and its recurrent state; the state sits in one block per
 *    request, is read from the zeroed trash block while the request has no
 *    past, and is overwritten in place; the packed batch runs as one row, with
 *    a varlen causal convolution continuing every sequence from its own conv
 *    state and the recurrence taking per-sequence states through cu_seqlens.
 *  - The gated delta rule (Yang, Kautz, Hatamizadeh, "Gated Delta Networks:
 *    Improving Mamba2 with Delta Rule", 2024, the gated delta rule equation):
 *        S_t = e^{g_t} S_{t-1} + beta_t (v_t - e^{g_t} S_{t-1} k_t) k_t^T,
 *        o_t = S_t q_t,
 *    with g_t = -exp(A_log) * softplus(a_t + dt_bias), beta_t = sigmoid(b_t),
 *    q and k L2-normalised and q scaled by 1/sqrt(d_k).
 *
 * A second rule, Kimi Delta Attention (KDA; the decay of the families the
 * "Continuous batching: model support tracker" page lists as Kimi Linear and
 * GLM5-next), keeps the same per-request states and the same convolution and
 * differs only in the gate: one decay per key channel instead of one per
 * head (Kimi Team, "Kimi Linear: An Expressive, Efficient Hybrid Linear
 * Attention Architecture", 2025, the KDA recurrence).  In the S[v][k]
 * orientation used here:
 *        S_t = S_{t-1} Diag(alpha_t) + beta_t (v_t - S_{t-1} Diag(alpha_t) k_t) k_t^T,
 *        o_t = S_t q_t,
 *    with alpha_t = exp(g_t), g_t[c] = -exp(A_log) * softplus(a_t[c] + dt_bias[c])
 *    for every key channel c (a_t and dt_bias have one entry per key channel).
 *
 * Everything is token by token in the order the definition states; there is
 * no chunking, blocking or reordering.  All arrays are fp64 and logical (no
 * pool byte layout here: the Python side converts).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - conv taps: w[c][K-1] multiplies the current token (PyTorch depthwise
 *    conv1d with padding K-1, first L outputs kept); no conv bias;
 *  - conv state = the last K-1 pre-convolution inputs, oldest row first;
 *  - L2 norm: x / sqrt(sum x^2 + 1e-6);
 *  - v-head h reads k-head h / (Hv/Hk);
 *  - channel order q | k | v, head-major inside each part.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_L2_EPS 1e-6

/* softplus(x) = log(1 + e^x), written so that e^x never overflows. */
static double softplus_f64(double x) {
  if (x > 0.0) return x + log1p(exp(-x));
  return log1p(exp(x));
}

static double sigmoid_f64(double x) {
  if (x >= 0.0) return 1.0 / (1.0 + exp(-x));
  double e = exp(x);
  return e / (1.0 + e);
}

static double silu_f64(double y) { return y * sigmoid_f64(y); }

/*
 * Varlen causal depthwise conv1d + SiLU for ONE sequence and a subset of
 * channels.
 *   x      : [L][C] this sequence's rows of the packed input (row stride C)
 *   tail   : [K-1][C] conv state (oldest first), read only
 *   w      : [C][K]
 *   ch0,nch: channel range to compute
 *   y      : [L][nch] output, SiLU applied
 * y_t[c] = SiLU( sum_{j=0}^{K-1} w[c][j] * xhat[t-K+1+j][c] ), where xhat is
 * the tail followed by the sequence's rows.
 */
void oracle_conv_silu_seq(int L, int C, int K, const double* x, const double* tail,
                          const double* w, int ch0, int nch, double* y) {
  for (int t = 0; t < L; ++t) {
    for (int c = ch0; c < ch0 + nch; ++c) {
      double acc = 0.0;
      for (int j = 0; j < K; ++j) {
        int p = t - (K - 1) + j; /* position in the sequence; <0 is the tail */
        double xv = (p >= 0) ? x[(size_t)p * C + c] : tail[(size_t)(K - 1 + p) * C + c];
        acc += w[(size_t)c * K + j] * xv;
      }
      y[(size_t)t * nch + (c - ch0)] = silu_f64(acc);
    }
  }
}

/* New conv state: the last K-1 rows of [old tail ; x_seq] (all channels). */
void oracle_conv_tail_update(int L, int C, int K, const double* x, const double* old_tail,
                             double* new_tail) {
  int W = K - 1;
  for (int r = 0; r < W; ++r) {
    int p = L - W + r; /* position in the sequence; <0 reaches into the old tail */
    for (int c = 0; c < C; ++c)
      new_tail[(size_t)r * C + c] = (p >= 0) ? x[(size_t)p * C + c] : old_tail[(size_t)(W + p) * C + c];
  }
}

/*
 * Gated delta rule for ONE (sequence, v-head) chain, given its per-token
 * inputs after the convolution.
 *   q,k : [L][dk] raw (SiLU output) rows of the k-head this v-head reads
 *   v   : [L][dv]
 *   graw: [L] gate pre-activation a_t (dt_bias and A_log applied here)
 *   braw: [L] b_t
 *   S   : [dv][dk] state, in: S_0, out: S_L (S[v][k])
 *   o   : [L][dv]
 */
void oracle_gdn_rule_head(int L, int dk, int dv, const double* q, const double* k, const double* v,
                          const double* a, const double* b, double A_log, double dt_bias,
                          double* S, double* o) {
  double* qn = (double*)malloc(sizeof(double) * dk);
  double* kn = (double*)malloc(sizeof(double) * dk);
  double* Sk = (double*)malloc(sizeof(double) * dv);
  for (int t = 0; t < L; ++t) {
    const double* qt = q + (size_t)t * dk;
    const double* kt = k + (size_t)t * dk;
    const double* vt = v + (size_t)t * dv;
    double sq = 0.0, sk = 0.0;
    for (int i = 0; i < dk; ++i) { sq += qt[i] * qt[i]; sk += kt[i] * kt[i]; }
    double qs = 1.0 / sqrt(sq + ORACLE_L2_EPS) / sqrt((double)dk);
    double ks = 1.0 / sqrt(sk + ORACLE_L2_EPS);
    for (int i = 0; i < dk; ++i) { qn[i] = qt[i] * qs; kn[i] = kt[i] * ks; }
    double g = -exp(A_log) * softplus_f64(a[t] + dt_bias);
    double beta = sigmoid_f64(b[t]);
    double decay = exp(g);
    /* S <- e^g S */
    for (int r = 0; r < dv * dk; ++r) S[r] *= decay;
    /* S <- S + beta (v - S k) k^T */
    for (int r = 0; r < dv; ++r) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(size_t)r * dk + i] * kn[i];
      Sk[r] = acc;
    }
    for (int r = 0; r < dv; ++r) {
      double u = beta * (vt[r] - Sk[r]);
      for (int i = 0; i < dk; ++i) S[(size_t)r * dk + i] += u * kn[i];
    }
    /* o = S q */
    for (int r = 0; r < dv; ++r) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(size_t)r * dk + i] * qn[i];
      o[(size_t)t * dv + r] = acc;
    }
  }
  free(qn); free(kn); free(Sk);
}

/*
 * KDA rule for ONE (sequence, v-head) chain: the gated delta rule with one
 * decay per key channel.  Arguments as oracle_gdn_rule_head, except
 *   a      : [L][dk] gate pre-activations, one per key channel
 *   dt_bias: [dk]
 * The decay scales column c (key channel c) of S[v][k] by alpha_t[c] before
 * the delta step; the delta step reads the decayed state.
 */
void oracle_kda_rule_head(int L, int dk, int dv, const double* q, const double* k, const double* v,
                          const double* a, const double* b, double A_log, const double* dt_bias,
                          double* S, double* o) {
  double* qn = (double*)malloc(sizeof(double) * dk);
  double* kn = (double*)malloc(sizeof(double) * dk);
  double* alpha = (double*)malloc(sizeof(double) * dk);
  double* Sk = (double*)malloc(sizeof(double) * dv);
  for (int t = 0; t < L; ++t) {
    const double* qt = q + (size_t)t * dk;
    const double* kt = k + (size_t)t * dk;
    const double* vt = v + (size_t)t * dv;
    double sq = 0.0, sk = 0.0;
    for (int i = 0; i < dk; ++i) { sq += qt[i] * qt[i]; sk += kt[i] * kt[i]; }
    double qs = 1.0 / sqrt(sq + ORACLE_L2_EPS) / sqrt((double)dk);
    double ks = 1.0 / sqrt(sk + ORACLE_L2_EPS);
    for (int i = 0; i < dk; ++i) { qn[i] = qt[i] * qs; kn[i] = kt[i] * ks; }
    for (int i = 0; i < dk; ++i)
      alpha[i] = exp(-exp(A_log) * softplus_f64(a[(size_t)t * dk + i] + dt_bias[i]));
    double beta = sigmoid_f64(b[t]);
    /* S <- S Diag(alpha): column i (key channel i) decays by alpha_i */
    for (int r = 0; r < dv; ++r)
      for (int i = 0; i < dk; ++i) S[(size_t)r * dk + i] *= alpha[i];
    /* S <- S + beta (v - S k) k^T */
    for (int r = 0; r < dv; ++r) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(size_t)r * dk + i] * kn[i];
      Sk[r] = acc;
    }
    for (int r = 0; r < dv; ++r) {
      double u = beta * (vt[r] - Sk[r]);
      for (int i = 0; i < dk; ++i) S[(size_t)r * dk + i] += u * kn[i];
    }
    /* o = S q */
    for (int r = 0; r < dv; ++r) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(size_t)r * dk + i] * qn[i];
      o[(size_t)t * dv + r] = acc;
    }
  }
  free(qn); free(kn); free(alpha); free(Sk);
}

/*
 * Whole packed forward, on logical fp64 arrays.
 *   x        : [T][C]  with C = 2*Hk*dk + Hv*dv
 *   a, b     : [T][Hv]
 *   cu       : [N+1] cumulative sequence starts
 *   blk      : [N] state block of each sequence (<0: padding, skipped)
 *   has_past : [N] 0 -> read block 0 (trash), else read blk
 *   w        : [C][K]; A_log, dt_bias: [Hv]
 *   conv_st  : [num_blocks][K-1][C] in/out
 *   rec_st   : [num_blocks][Hv][dv][dk] in/out (S[v][k], logical; the Python
 *              side maps it to the pool's k-major byte layout)
 *   out      : [T][Hv][dv]; rows of skipped sequences are left untouched
 *   skip     : [N] or NULL: nonzero entries are skipped like padding (data
 *              errors found by the caller's validation)
 * Returns the number of OpenMP threads used.
 *
 * gate_width is 1 for the gated delta rule (a [T][Hv], dt_bias [Hv]) and dk
 * for KDA (a [T][Hv][dk], dt_bias [Hv][dk]); nothing else differs.
 */
static int packed_forward(int T, int N, int Hk, int Hv, int dk, int dv, int K, int num_blocks,
                          const double* x, const double* a, const double* b, const int32_t* cu,
                          const int32_t* blk, const uint8_t* has_past, const uint8_t* skip,
                          const double* w, const double* A_log, const double* dt_bias,
                          double* conv_st, double* rec_st, double* out, int nthreads,
                          int gate_width) {
  (void)T;
  const int C = 2 * Hk * dk + Hv * dv;
  const int W = K - 1;
  const int ratio = Hv / Hk;
  const size_t conv_blk = (size_t)W * C;
  const size_t rec_head = (size_t)dv * dk;
  const size_t rec_blk = (size_t)Hv * rec_head;
  int used = 1;
  (void)num_blocks;

  /* Phase 1: every (sequence, v-head) chain reads its source block and
   * computes its outputs and final state into private buffers. */
  int npairs = N * Hv;
  double** Sfin = (double**)calloc((size_t)npairs, sizeof(double*));
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
    int s = pair / Hv, h = pair % Hv;
    int L = cu[s + 1] - cu[s];
    if (blk[s] < 0 || L <= 0 || (skip && skip[s])) continue;
    int src = has_past[s] ? blk[s] : 0;
    int kh = h / ratio;
    const double* xs = x + (size_t)cu[s] * C;
    const double* tail = conv_st + (size_t)src * conv_blk;
    double* qy = (double*)malloc(sizeof(double) * (size_t)L * dk);
    double* ky = (double*)malloc(sizeof(double) * (size_t)L * dk);
    double* vy = (double*)malloc(sizeof(double) * (size_t)L * dv);
    double* at = (double*)malloc(sizeof(double) * (size_t)L * gate_width);
    double* bt = (double*)malloc(sizeof(double) * (size_t)L);
    double* o = (double*)malloc(sizeof(double) * (size_t)L * dv);
    double* S = (double*)malloc(sizeof(double) * rec_head);
    oracle_conv_silu_seq(L, C, K, xs, tail, w, kh * dk, dk, qy);
    oracle_conv_silu_seq(L, C, K, xs, tail, w, Hk * dk + kh * dk, dk, ky);
    oracle_conv_silu_seq(L, C, K, xs, tail, w, 2 * Hk * dk + h * dv, dv, vy);
    for (int t = 0; t < L; ++t) {
      for (int c = 0; c < gate_width; ++c)
        at[(size_t)t * gate_width + c] = a[((size_t)(cu[s] + t) * Hv + h) * gate_width + c];
      bt[t] = b[(size_t)(cu[s] + t) * Hv + h];
    }
    memcpy(S, rec_st + (size_t)src * rec_blk + (size_t)h * rec_head, sizeof(double) * rec_head);
    if (gate_width == 1)
      oracle_gdn_rule_head(L, dk, dv, qy, ky, vy, at, bt, A_log[h], dt_bias[h], S, o);
    else
      oracle_kda_rule_head(L, dk, dv, qy, ky, vy, at, bt, A_log[h], dt_bias + (size_t)h * dk, S, o);
    for (int t = 0; t < L; ++t)
      memcpy(out + ((size_t)(cu[s] + t) * Hv + h) * dv, o + (size_t)t * dv, sizeof(double) * dv);
    Sfin[pair] = S;
    free(qy); free(ky); free(vy); free(at); free(bt); free(o);
  }

  /* Phase 2: new conv tails, computed from the source blocks before any
   * block is overwritten. */
  double** tails = (double**)calloc((size_t)N, sizeof(double*));
  for (int s = 0; s < N; ++s) {
    int L = cu[s + 1] - cu[s];
    if (blk[s] < 0 || L <= 0 || (skip && skip[s])) continue;
    int src = has_past[s] ? blk[s] : 0;
    tails[s] = (double*)malloc(sizeof(double) * conv_blk);
    oracle_conv_tail_update(L, C, K, x + (size_t)cu[s] * C, conv_st + (size_t)src * conv_blk, tails[s]);
  }

  /* Phase 3: overwrite each request's block in place. */
  for (int s = 0; s < N; ++s) {
    if (!tails[s]) continue;
    memcpy(conv_st + (size_t)blk[s] * conv_blk, tails[s], sizeof(double) * conv_blk);
    free(tails[s]);
    for (int h = 0; h < Hv; ++h) {
      double* S = Sfin[s * Hv + h];
      memcpy(rec_st + (size_t)blk[s] * rec_blk + (size_t)h * rec_head, S, sizeof(double) * rec_head);
      free(S);
    }
  }
  free(tails);
  free(Sfin);
  return used;
}

int oracle_gdn_forward(int T, int N, int Hk, int Hv, int dk, int dv, int K, int num_blocks,
                       const double* x, const double* a, const double* b, const int32_t* cu,
                       const int32_t* blk, const uint8_t* has_past, const uint8_t* skip,
                       const double* w, const double* A_log, const double* dt_bias,
                       double* conv_st, double* rec_st, double* out, int nthreads) {
  return packed_forward(T, N, Hk, Hv, dk, dv, K, num_blocks, x, a, b, cu, blk, has_past, skip, w,
                        A_log, dt_bias, conv_st, rec_st, out, nthreads, 1);
}

/* The same packed forward with the KDA rule: a [T][Hv][dk], dt_bias [Hv][dk]. */
int oracle_kda_forward(int T, int N, int Hk, int Hv, int dk, int dv, int K, int num_blocks,
                       const double* x, const double* a, const double* b, const int32_t* cu,
                       const int32_t* blk, const uint8_t* has_past, const uint8_t* skip,
                       const double* w, const double* A_log, const double* dt_bias,
                       double* conv_st, double* rec_st, double* out, int nthreads) {
  return packed_forward(T, N, Hk, Hv, dk, dv, K, num_blocks, x, a, b, cu, blk, has_past, skip, w,
                        A_log, dt_bias, conv_st, rec_st, out, nthreads, dk);
}
