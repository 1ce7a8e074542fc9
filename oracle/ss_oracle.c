/*
 * CPU oracle for the selective state-space scan (S6) — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, sequential float64 restatement of what the selective scan
 * computes. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this library; the product path never does.
 *
 * Definition followed (float64 throughout, inputs widened exactly):
 *   for each batch b and channel d, with h_n <- h0[b,d,n] (0 when absent),
 *   for t = 0 .. L-1:
 *     delta = softplus(delta_raw[b,t,d] + bias[d])
 *     for each state n:
 *       h_n = exp(delta * A[d,n]) * h_n + delta * B[b,t,n] * u[b,t,d]
 *     y   = sum_n C[b,t,n] * h_n + D[d] * u[b,t,d]
 *     out[b,t,d] = y * z / (1 + exp(-z))        (z = z[b,t,d], when z is given)
 *   h_last[b,d,n] = h_n after the last step.
 *
 * Sources (page titles and sections):
 *  - discretised recurrence h_t = Abar h_{t-1} + Bbar x_t, y_t = C h_t + D x_t:
 *    "Transformer时代终结？Mamba的状态空间革命重塑AI底层架构", section 二.1
 *    (continuous system and its discretisation);
 *  - Abar = exp(delta*A) (zero-order hold) and the first-order Bbar ~= delta*B:
 *    "外文文献精读：Mamba - 线性时间序列建模与结构化状态空间模型", section 1.2,
 *    and the mlqm.cn SSM tutorial (untitled in the capture), section 3.2
 *    (discretisation) and the section 9.2 step sketch, which computes
 *    dA = exp(dt*A), dB = dt*B and y = (h*C).sum + D*x;
 *  - delta, B, C as functions of the input, B and C shared by all channels:
 *    mlqm.cn tutorial, sections 5.2 and 9.2 (Bk, Ck have shape (d_state,));
 *  - A = -exp(A_log): "外文文献精读" page, section 4.1 (stability);
 *  - SiLU output gate: review page ("Mamba: Linear-Time Sequence Modeling with
 *    Selective State Spaces"), method step 3, and mlqm.cn tutorial section 7.1;
 *  - softplus for delta: not printed on the pages; taken as
 *    softplus(x) = log(1 + e^x), evaluated without overflow;
 *  - single-token decode = the same step with L = 1 and h carried in place:
 *    "AI 推理系列（十四）：Mamba 的 Selective State Space", section
 *    "Selective Scan 如何兼顾训练与 Decode".
 *
 * Parity pins live in the tests (brute-force unrolled sum, LTI convolution,
 * delta->0, large delta, chunk associativity, closed forms).
 *
 * The file also holds the gradients of the scan (ss_oracle_scan_bwd, pinned by
 * central finite differences of the forward oracle), and the block's causal
 * depthwise convolution front-end and
 * its decode step (ss_oracle_conv1d, ss_oracle_conv1d_update, at the end),
 * pinned against numpy's convolution, impulse responses, chunk continuity and
 * decode-equals-forward; and the generalised scan (ss_oracle_scan_general: any
 * state size, grouped B and C, zero-order-hold Bbar), pinned against scipy's
 * zero-order-hold discretisation and simulation of the same linear system, the
 * scan above on its special case, per-group slices and a split of the states.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype codes of the raw input arrays */
#define ORC_F32 0
#define ORC_BF16 1

static double widen(const void *p, int dtype, int64_t i) {
  if (dtype == ORC_F32) return (double)((const float *)p)[i];
  /* bfloat16: the upper 16 bits of an IEEE binary32 value */
  uint32_t bits = (uint32_t)((const uint16_t *)p)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static double softplus(double x) {
  /* log(1 + e^x) without overflow: for x > 0 use x + log(1 + e^-x) */
  if (x > 0) return x + log1p(exp(-x));
  return log1p(exp(x));
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

typedef struct {
  int64_t batch, seqlen, dim, dstate;
  int in_dtype;
  const void *u, *delta_raw, *z, *B, *C;
  const float *A, *Dskip, *bias, *h0;
  const int64_t *chans; /* (b, d) pairs, 2 per channel */
  int64_t n_chan;
  double *y;      /* [n_chan][seqlen] */
  double *h_last; /* [n_chan][dstate] */
  int64_t next;   /* work counter */
  pthread_mutex_t mu;
} scan_job;

static void scan_one(const scan_job *j, int64_t c) {
  const int64_t L = j->seqlen, Dm = j->dim, N = j->dstate;
  const int64_t b = j->chans[2 * c], d = j->chans[2 * c + 1];
  double *h = (double *)malloc(sizeof(double) * (size_t)N);
  for (int64_t n = 0; n < N; n++) h[n] = j->h0 ? (double)j->h0[(b * Dm + d) * N + n] : 0.0;
  const double bias = j->bias ? (double)j->bias[d] : 0.0;
  const double dsk = j->Dskip ? (double)j->Dskip[d] : 0.0;
  for (int64_t t = 0; t < L; t++) {
    const int64_t i = (b * L + t) * Dm + d;     /* [b][t][d] */
    const int64_t r = (b * L + t) * N;          /* [b][t][n] row */
    const double delta = softplus(widen(j->delta_raw, j->in_dtype, i) + bias);
    const double x = widen(j->u, j->in_dtype, i);
    double y = 0.0;
    for (int64_t n = 0; n < N; n++) {
      const double abar = exp(delta * (double)j->A[d * N + n]);
      const double bbar_x = delta * widen(j->B, j->in_dtype, r + n) * x;
      h[n] = abar * h[n] + bbar_x;
      y += widen(j->C, j->in_dtype, r + n) * h[n];
    }
    y += dsk * x;
    if (j->z) y *= silu(widen(j->z, j->in_dtype, i));
    j->y[c * L + t] = y;
  }
  for (int64_t n = 0; n < N; n++) j->h_last[c * N + n] = h[n];
  free(h);
}

static void *scan_worker(void *arg) {
  scan_job *j = (scan_job *)arg;
  for (;;) {
    pthread_mutex_lock(&j->mu);
    int64_t c = j->next++;
    pthread_mutex_unlock(&j->mu);
    if (c >= j->n_chan) break;
    scan_one(j, c);
  }
  return NULL;
}

/*
 * Selective scan over the channels listed in `chans` ((b, d) pairs).
 * u, delta_raw, z: [batch][seqlen][dim]; B, C: [batch][seqlen][dstate] in
 * in_dtype; A: [dim][dstate]; Dskip, bias: [dim] or NULL; h0:
 * [batch][dim][dstate] or NULL; z NULL means no gate.
 * Writes y[c][t] and h_last[c][n] for listed channel c. Returns 0, or -1 on
 * a bad argument.
 */
int ss_oracle_scan(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int in_dtype,
                   const void *u, const void *delta_raw, const void *z, const void *B,
                   const void *C, const float *A, const float *Dskip, const float *bias,
                   const float *h0, const int64_t *chans, int64_t n_chan, double *y,
                   double *h_last, int nthreads) {
  if (batch < 0 || seqlen < 0 || dim < 0 || dstate <= 0 || n_chan < 0) return -1;
  if (in_dtype != ORC_F32 && in_dtype != ORC_BF16) return -1;
  if (!u || !delta_raw || !B || !C || !A || !chans || !y || !h_last) return -1;
  for (int64_t c = 0; c < n_chan; c++)
    if (chans[2 * c] < 0 || chans[2 * c] >= batch || chans[2 * c + 1] < 0 || chans[2 * c + 1] >= dim)
      return -1;
  scan_job j;
  memset(&j, 0, sizeof j);
  j.batch = batch; j.seqlen = seqlen; j.dim = dim; j.dstate = dstate; j.in_dtype = in_dtype;
  j.u = u; j.delta_raw = delta_raw; j.z = z; j.B = B; j.C = C;
  j.A = A; j.Dskip = Dskip; j.bias = bias; j.h0 = h0;
  j.chans = chans; j.n_chan = n_chan; j.y = y; j.h_last = h_last; j.next = 0;
  pthread_mutex_init(&j.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int k = 1; k < nthreads; k++)
    if (pthread_create(&th[started], NULL, scan_worker, &j) == 0) started++;
  scan_worker(&j);
  for (int k = 0; k < started; k++) pthread_join(th[k], NULL);
  pthread_mutex_destroy(&j.mu);
  return 0;
}

/*
 * One decode step for the listed channels, state carried in place:
 * h: [batch][dim][dstate] float64, updated; u, delta_raw, z: [batch][dim];
 * B, C: [batch][dstate]; writes y[c] for listed channel c.
 */
int ss_oracle_state_update(int64_t batch, int64_t dim, int64_t dstate, int in_dtype, double *h,
                           const void *u, const void *delta_raw, const void *z, const void *B,
                           const void *C, const float *A, const float *Dskip, const float *bias,
                           const int64_t *chans, int64_t n_chan, double *y) {
  if (batch < 0 || dim < 0 || dstate <= 0 || n_chan < 0) return -1;
  if (in_dtype != ORC_F32 && in_dtype != ORC_BF16) return -1;
  if (!h || !u || !delta_raw || !B || !C || !A || !chans || !y) return -1;
  for (int64_t c = 0; c < n_chan; c++) {
    const int64_t b = chans[2 * c], d = chans[2 * c + 1];
    if (b < 0 || b >= batch || d < 0 || d >= dim) return -1;
    const int64_t i = b * dim + d;
    const double delta = softplus(widen(delta_raw, in_dtype, i) + (bias ? (double)bias[d] : 0.0));
    const double x = widen(u, in_dtype, i);
    double *hs = h + i * dstate;
    double acc = 0.0;
    for (int64_t n = 0; n < dstate; n++) {
      hs[n] = exp(delta * (double)A[d * dstate + n]) * hs[n] +
              delta * widen(B, in_dtype, b * dstate + n) * x;
      acc += widen(C, in_dtype, b * dstate + n) * hs[n];
    }
    acc += (Dskip ? (double)Dskip[d] : 0.0) * x;
    if (z) acc *= silu(widen(z, in_dtype, i));
    y[c] = acc;
  }
  return 0;
}

/*
 * Causal depthwise 1-D convolution of the Mamba block's front-end, with SiLU.
 *
 * The block feeds the expanded input through a short causal convolution along
 * the sequence and a SiLU before the selective SSM ("Mamba: Linear-Time
 * Sequence Modeling with Selective State Spaces" review page, method step 3;
 * mlqm.cn tutorial section 7.1, the block diagram). Decoding keeps, per
 * request, the few past inputs that convolution needs ("AI 推理系列（十四）：
 * Mamba 的 Selective State Space", the decode-state table and the sections on
 * the request state). The pages give no kernel width, tap order or bias; the
 * reading taken here, for each batch b and channel d, with width K:
 *   e[p] = x[b,p,d] for p >= 0, state_in[b,d,p+K-1] for -(K-1) <= p < 0
 *          (0 when state_in is NULL)
 *   pre  = bias[d] + sum_{k<K} w[d,k] * e[t-(K-1)+k]
 *   y[b,t,d] = silu(pre) when silu_on, else pre
 *   state_out[b,d,k] = e[L-(K-1)+k] for k < K-1   (the last K-1 inputs)
 * x, state_in: in_dtype; w: [dim][K]; bias: [dim] or NULL.
 * y: [batch][seqlen][dim] float64; state_out: [batch][dim][K-1] float64 or NULL.
 */
int ss_oracle_conv1d(int64_t batch, int64_t seqlen, int64_t dim, int64_t width, int in_dtype,
                     const void *x, const float *w, const float *bias, const void *state_in,
                     int silu_on, double *y, double *state_out) {
  if (batch < 0 || seqlen < 0 || dim < 0 || width < 1) return -1;
  if (in_dtype != ORC_F32 && in_dtype != ORC_BF16) return -1;
  if (!x || !w || !y) return -1;
  const int64_t H = width - 1;
  double *e = (double *)malloc(sizeof(double) * (size_t)(seqlen + H + 1));
  if (!e) return -1;
  for (int64_t b = 0; b < batch; b++) {
    for (int64_t d = 0; d < dim; d++) {
      /* e[q] holds position p = q - H */
      for (int64_t q = 0; q < H; q++)
        e[q] = state_in ? widen(state_in, in_dtype, (b * dim + d) * H + q) : 0.0;
      for (int64_t t = 0; t < seqlen; t++) e[H + t] = widen(x, in_dtype, (b * seqlen + t) * dim + d);
      for (int64_t t = 0; t < seqlen; t++) {
        double pre = bias ? (double)bias[d] : 0.0;
        for (int64_t k = 0; k < width; k++) pre += (double)w[d * width + k] * e[t + k];
        y[(b * seqlen + t) * dim + d] = silu_on ? silu(pre) : pre;
      }
      if (state_out)
        for (int64_t k = 0; k < H; k++) state_out[(b * dim + d) * H + k] = e[seqlen + k];
    }
  }
  free(e);
  return 0;
}

/*
 * One decode step of the convolution, state carried in place: state
 * [batch][dim][K-1] float64 holds the last K-1 inputs, oldest first; x
 * [batch][dim] in in_dtype is the new input. y = silu(bias + sum_{k<K-1}
 * w[d,k] state[k] + w[d,K-1] x), then the state drops its oldest entry and
 * appends x.
 */
int ss_oracle_conv1d_update(int64_t batch, int64_t dim, int64_t width, int in_dtype, double *state,
                            const void *x, const float *w, const float *bias, int silu_on, double *y) {
  if (batch < 0 || dim < 0 || width < 1) return -1;
  if (in_dtype != ORC_F32 && in_dtype != ORC_BF16) return -1;
  if (!x || !w || !y || (width > 1 && !state)) return -1;
  const int64_t H = width - 1;
  for (int64_t b = 0; b < batch; b++) {
    for (int64_t d = 0; d < dim; d++) {
      double *s = state ? state + (b * dim + d) * H : NULL;
      const double xv = widen(x, in_dtype, b * dim + d);
      double pre = bias ? (double)bias[d] : 0.0;
      for (int64_t k = 0; k < H; k++) pre += (double)w[d * width + k] * s[k];
      pre += (double)w[d * width + H] * xv;
      y[b * dim + d] = silu_on ? silu(pre) : pre;
      for (int64_t k = 0; k + 1 < H; k++) s[k] = s[k + 1];
      if (H > 0) s[H - 1] = xv;
    }
  }
  return 0;
}

/*
 * Gradients of the selective scan (the backward pass), by the reverse sweep of
 * the adjoint state, in float64. The pages train Mamba end to end and say the
 * backward pass recomputes the forward states instead of storing them (review
 * page, method step 2 (3); "AI 推理系列（十四）", training section); the
 * gradients themselves follow from differentiating the recurrence the header
 * defines. For each channel (b, d), with dyv_t = dy_t * g_t, g_t = silu(z_t)
 * (1 when z is NULL) and yv_t = sum_n C_t,n h_t,n + D u_t:
 *   lambda_{L-1} = C_{L-1} dyv_{L-1} + dh_last
 *   lambda_t     = C_t dyv_t + Abar_{t+1} lambda_{t+1}          (per state n)
 *   dB[b,t,n]   += lambda_t,n delta_t u_t        (summed over channels d)
 *   dC[b,t,n]   += dyv_t h_t,n                   (summed over channels d)
 *   du_t         = dyv_t D + delta_t sum_n lambda_t,n B_t,n
 *   ddelta_t     = sum_n lambda_t,n (h_{t-1},n Abar_t,n A_n + B_t,n u_t)
 *   dA[d,n]     += lambda_t,n h_{t-1},n Abar_t,n delta_t
 *   dD[d]       += dyv_t u_t
 *   dz_t         = dy_t yv_t silu'(z_t),  silu'(z) = s (1 + z (1 - s)), s = sigmoid(z)
 *   ddelta_raw_t = ddelta_t sigmoid(delta_raw_t + bias_d);   dbias[d] += ddelta_raw_t
 *   dh0[b,d,n]   = Abar_0,n lambda_0,n
 * dy: [batch][seqlen][dim] in dy_dtype; dh_last, h0: [batch][dim][dstate] or NULL.
 * Outputs (float64, overwritten): du, ddelta_raw, dz [batch][seqlen][dim]; dA
 * [dim][dstate]; dB, dC [batch][seqlen][dstate]; dD, dbias [dim]; dh0
 * [batch][dim][dstate]. Single-threaded (the reductions over channels).
 */
static double dsilu(double z) {
  const double s = 1.0 / (1.0 + exp(-z));
  return s * (1.0 + z * (1.0 - s));
}

int ss_oracle_scan_bwd(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int in_dtype, int dy_dtype,
                       const void *u, const void *delta_raw, const void *z, const void *B, const void *C,
                       const float *A, const float *Dskip, const float *bias, const float *h0, const void *dy,
                       const float *dh_last, double *du, double *ddelta_raw, double *dz, double *dA, double *dB,
                       double *dC, double *dD, double *dbias, double *dh0) {
  if (batch < 0 || seqlen < 0 || dim < 0 || dstate <= 0) return -1;
  if ((in_dtype != ORC_F32 && in_dtype != ORC_BF16) || (dy_dtype != ORC_F32 && dy_dtype != ORC_BF16)) return -1;
  if (!u || !delta_raw || !B || !C || !A || !dy || !du || !ddelta_raw || !dz || !dA || !dB || !dC || !dD ||
      !dbias || !dh0)
    return -1;
  const int64_t L = seqlen, Dm = dim, N = dstate;
  memset(dA, 0, sizeof(double) * (size_t)(Dm * N));
  memset(dB, 0, sizeof(double) * (size_t)(batch * L * N));
  memset(dC, 0, sizeof(double) * (size_t)(batch * L * N));
  memset(dD, 0, sizeof(double) * (size_t)Dm);
  memset(dbias, 0, sizeof(double) * (size_t)Dm);
  double *hist = (double *)malloc(sizeof(double) * (size_t)((L + 1) * N)); /* hist[t+1] = h_t, hist[0] = h0 */
  double *lam = (double *)malloc(sizeof(double) * (size_t)N);
  double *delta = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  if (!hist || !lam || !delta) {
    free(hist);
    free(lam);
    free(delta);
    return -1;
  }
  for (int64_t b = 0; b < batch; b++) {
    for (int64_t d = 0; d < Dm; d++) {
      const double bs = bias ? (double)bias[d] : 0.0;
      const double dsk = Dskip ? (double)Dskip[d] : 0.0;
      /* forward, keeping every state */
      for (int64_t n = 0; n < N; n++) hist[n] = h0 ? (double)h0[(b * Dm + d) * N + n] : 0.0;
      for (int64_t t = 0; t < L; t++) {
        const int64_t i = (b * L + t) * Dm + d, r = (b * L + t) * N;
        delta[t] = softplus(widen(delta_raw, in_dtype, i) + bs);
        const double x = widen(u, in_dtype, i);
        for (int64_t n = 0; n < N; n++)
          hist[(t + 1) * N + n] = exp(delta[t] * (double)A[d * N + n]) * hist[t * N + n] +
                                  delta[t] * widen(B, in_dtype, r + n) * x;
      }
      /* reverse sweep of the adjoint state */
      for (int64_t n = 0; n < N; n++) lam[n] = dh_last ? (double)dh_last[(b * Dm + d) * N + n] : 0.0;
      for (int64_t t = L - 1; t >= 0; t--) {
        const int64_t i = (b * L + t) * Dm + d, r = (b * L + t) * N;
        const double x = widen(u, in_dtype, i);
        const double dyt = widen(dy, dy_dtype, i);
        const double zz = z ? widen(z, in_dtype, i) : 0.0;
        const double g = z ? silu(zz) : 1.0;
        const double dyv = dyt * g;
        double yv = dsk * x;
        for (int64_t n = 0; n < N; n++) yv += widen(C, in_dtype, r + n) * hist[(t + 1) * N + n];
        double dut = dyv * dsk, ddel = 0.0;
        for (int64_t n = 0; n < N; n++) {
          const double a = exp(delta[t] * (double)A[d * N + n]);
          const double Bn = widen(B, in_dtype, r + n), Cn = widen(C, in_dtype, r + n);
          /* lambda_t = C_t dyv_t + (already folded) Abar_{t+1} lambda_{t+1} */
          lam[n] += Cn * dyv;
          dC[r + n] += dyv * hist[(t + 1) * N + n];
          dB[r + n] += lam[n] * delta[t] * x;
          dut += lam[n] * delta[t] * Bn;
          ddel += lam[n] * (hist[t * N + n] * a * (double)A[d * N + n] + Bn * x);
          dA[d * N + n] += lam[n] * hist[t * N + n] * a * delta[t];
          lam[n] *= a; /* becomes Abar_t lambda_t, the carry into step t-1 */
        }
        dD[d] += dyv * x;
        du[i] = dut;
        dz[i] = z ? dyt * yv * dsilu(zz) : 0.0;
        const double sg = 1.0 / (1.0 + exp(-(widen(delta_raw, in_dtype, i) + bs)));
        ddelta_raw[i] = ddel * sg;
        dbias[d] += ddel * sg;
      }
      for (int64_t n = 0; n < N; n++) dh0[(b * Dm + d) * N + n] = lam[n]; /* Abar_0 lambda_0 */
    }
  }
  free(hist);
  free(lam);
  free(delta);
  return 0;
}

/*
 * Generalised selective scan: any state size N, B and C shared within G groups
 * of channels, and the zero-order-hold input matrix as an alternative to the
 * first-order one.
 *
 *  - state size: the pages' tutorial lets the state dimension N grow (16 in the
 *    paper's language models, larger for other modalities; mlqm.cn tutorial,
 *    section 3.1); nothing in the recurrence depends on N;
 *  - zero-order hold: the exact discretisation of h' = A h + B x for an input
 *    held constant over a step of length delta gives
 *      Abar = exp(delta A),  Bbar = (exp(delta A) - 1) / A * B
 *    for diagonal A ("外文文献精读" page, section 1.2; tutorial section 3.2),
 *    which tends to delta B as delta A -> 0 (the first-order form the scan
 *    above uses);
 *  - groups: B and C are produced per token for G groups of dim / G consecutive
 *    channels each; channel d reads group d / (dim / G) (G = 1: shared by all
 *    channels, G = dim: one B and C per channel). The pages give one shared
 *    B and C; grouping is the plainest generalisation of that sharing.
 *
 * B, C: [batch][seqlen][G][N]; A: [dim][N]; everything else as ss_oracle_scan.
 * disc: 0 = first order (Bbar = delta B), 1 = zero-order hold. For A[d,n] = 0
 * the zero-order hold Bbar is delta B (its limit).
 * Writes y[c][t] and h_last[c][n] for listed channel c. Returns 0, or -1 on a
 * bad argument (including dim not divisible by G).
 */
typedef struct {
  int64_t batch, seqlen, dim, dstate, ngroups;
  int disc, in_dtype;
  const void *u, *delta_raw, *z, *B, *C;
  const float *A, *Dskip, *bias, *h0;
  const int64_t *chans;
  int64_t n_chan;
  double *y, *h_last;
  int64_t next;
  pthread_mutex_t mu;
} gscan_job;

static void gscan_one(const gscan_job *j, int64_t c) {
  const int64_t L = j->seqlen, Dm = j->dim, N = j->dstate, G = j->ngroups;
  const int64_t b = j->chans[2 * c], d = j->chans[2 * c + 1];
  const int64_t g = d / (Dm / G);
  double *h = (double *)malloc(sizeof(double) * (size_t)N);
  for (int64_t n = 0; n < N; n++) h[n] = j->h0 ? (double)j->h0[(b * Dm + d) * N + n] : 0.0;
  const double bias = j->bias ? (double)j->bias[d] : 0.0;
  const double dsk = j->Dskip ? (double)j->Dskip[d] : 0.0;
  for (int64_t t = 0; t < L; t++) {
    const int64_t i = (b * L + t) * Dm + d;        /* [b][t][d] */
    const int64_t r = ((b * L + t) * G + g) * N;   /* [b][t][g][n] row */
    const double delta = softplus(widen(j->delta_raw, j->in_dtype, i) + bias);
    const double x = widen(j->u, j->in_dtype, i);
    double y = 0.0;
    for (int64_t n = 0; n < N; n++) {
      const double a = (double)j->A[d * N + n];
      const double abar = exp(delta * a);
      /* the factor that multiplies B: delta (first order) or expm1(delta a) / a */
      const double bfac = (j->disc == 1 && a != 0.0) ? expm1(delta * a) / a : delta;
      h[n] = abar * h[n] + bfac * widen(j->B, j->in_dtype, r + n) * x;
      y += widen(j->C, j->in_dtype, r + n) * h[n];
    }
    y += dsk * x;
    if (j->z) y *= silu(widen(j->z, j->in_dtype, i));
    j->y[c * L + t] = y;
  }
  for (int64_t n = 0; n < N; n++) j->h_last[c * N + n] = h[n];
  free(h);
}

static void *gscan_worker(void *arg) {
  gscan_job *j = (gscan_job *)arg;
  for (;;) {
    pthread_mutex_lock(&j->mu);
    int64_t c = j->next++;
    pthread_mutex_unlock(&j->mu);
    if (c >= j->n_chan) break;
    gscan_one(j, c);
  }
  return NULL;
}

int ss_oracle_scan_general(int64_t batch, int64_t seqlen, int64_t dim, int64_t dstate, int64_t ngroups,
                           int disc, int in_dtype, const void *u, const void *delta_raw, const void *z,
                           const void *B, const void *C, const float *A, const float *Dskip, const float *bias,
                           const float *h0, const int64_t *chans, int64_t n_chan, double *y, double *h_last,
                           int nthreads) {
  if (batch < 0 || seqlen < 0 || dim < 0 || dstate <= 0 || n_chan < 0 || ngroups <= 0) return -1;
  if (dim % ngroups != 0 || (disc != 0 && disc != 1)) return -1;
  if (in_dtype != ORC_F32 && in_dtype != ORC_BF16) return -1;
  if (!u || !delta_raw || !B || !C || !A || !chans || !y || !h_last) return -1;
  for (int64_t c = 0; c < n_chan; c++)
    if (chans[2 * c] < 0 || chans[2 * c] >= batch || chans[2 * c + 1] < 0 || chans[2 * c + 1] >= dim)
      return -1;
  gscan_job j;
  memset(&j, 0, sizeof j);
  j.batch = batch; j.seqlen = seqlen; j.dim = dim; j.dstate = dstate; j.ngroups = ngroups;
  j.disc = disc; j.in_dtype = in_dtype;
  j.u = u; j.delta_raw = delta_raw; j.z = z; j.B = B; j.C = C;
  j.A = A; j.Dskip = Dskip; j.bias = bias; j.h0 = h0;
  j.chans = chans; j.n_chan = n_chan; j.y = y; j.h_last = h_last; j.next = 0;
  pthread_mutex_init(&j.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  int started = 0;
  for (int k = 1; k < nthreads; k++)
    if (pthread_create(&th[started], NULL, gscan_worker, &j) == 0) started++;
  gscan_worker(&j);
  for (int k = 0; k < started; k++) pthread_join(th[k], NULL);
  pthread_mutex_destroy(&j.mu);
  return 0;
}
