/*
 * fp64 CPU oracle for the selective-scan forward, its gradients (backward) and the
 * recurrent decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark may load this library.  It shares no
 * code, header, table or helper with the CUDA library it is used to check.
 *
 * What it computes (plain definition, sequential in t, fp64 throughout):
 *
 *   for every batch b and channel d, with h[n] = h0[b,d,n] (or 0):
 *     for t = 0 .. L-1:
 *       x      = delta[b,d,t] + delta_bias[d]
 *       Δ      = softplus(x) = log(1 + e^x)     if delta_softplus, else x
 *       for n: h[n] = exp(Δ·A[d,n])·h[n] + Δ·B[b,n,t]·u[b,d,t]
 *       y      = Σ_n C[b,n,t]·h[n] + D[d]·u[b,d,t]
 *       out[b,d,t] = y · z·σ(z)  with z = z[b,d,t]   (y unchanged without z)
 *     h_last[b,d,:] = h
 *
 * Sources (pages on the Mamba selective SSM):
 *  - "Mamba状态空间模型深度解析：挑战Transformer的下一代序列建模范式" §2.1: the
 *    selective recurrence h_k = A·h_{k-1} + B(x_k)·x_k, y_k = C(x_k)·h_k, with
 *    B, C and Δ functions of the input; y_k reads the state after step k.
 *  - "Mamba架构与SSM模型：高效序列建模技术解析" §2.1: zero-order-hold
 *    Ā = exp(ΔA); §2.2: Δ = softplus(Linear(x) + param_Δ).  The Linear layer
 *    is upstream of this operation, so its output arrives as `delta`.
 *  - "Mamba: Linear-Time Sequence Modeling with Selective SSMs", "连续与离散SSM":
 *    the D·u feed-through term of y = Cx + Du.
 *  - "Mamba状态空间模型深度解析" §3.1: SiLU multiplicative gate in the block.
 *  - "Mamba: Linear-Time Sequence Modeling with Selective SSMs", "选择性扫描要点":
 *    the end state of one block is carried as the start ("prefix") state of
 *    the next, which is what h0 / h_last expose.
 *
 * Readings where the pages leave a step open:
 *  - B̄ is taken as Δ·B (the simplified discretisation of the input matrix).
 *    With `zoh` it is the exact zero-order-hold form (ΔA)^{-1}(exp(ΔA)-I)·ΔB
 *    that "Mamba架构与SSM模型：高效序列建模技术解析" §2.1 prints; for the
 *    diagonal A this is (exp(ΔA_n) - 1)/A_n · B_n per state, Δ·B_n at A_n = 0.
 *  - `reverse` runs the same recurrence from t = L-1 down to 0 (the backward
 *    direction of a bidirectional layer): h_t = Ā_t·h_{t+1} + B̄_t·u_t.
 *  - The gate multiplies the whole y, including the D·u term.
 *  - softplus is the exact log(1+e^x), evaluated as max(x,0) + log1p(e^{-|x|}).
 *  - silu(z) = z / (1 + e^{-z}).
 *
 * Inputs are read as the exact values of their stored type: fp32 as is, bf16
 * (raw 16-bit patterns) widened exactly.  Results are fp64.
 *
 * Build: gcc -O2 -std=c11 -shared -fPIC -pthread selscan_oracle.c -lm
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* dtype codes of the input tensors u, delta, z, B, C */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* Exact widening of one stored input element to double. */
static double load_in(const void* p, int64_t i, int dtype) {
  if (dtype == ORACLE_BF16) {
    uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float*)p)[i];
}

static double softplus(double x) {
  return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

typedef struct {
  int64_t batch, dim, seqlen, dstate;
  int in_dtype;
  const void *u, *delta, *z, *B, *C;
  const float *A, *D, *delta_bias, *h0;
  const double* h0_f64; /* fp64 start state; takes precedence over h0 */
  const double* u_f64;  /* fp64 input [B, D, L]; takes precedence over u */
  int delta_softplus;
  int reverse; /* process t from L-1 down to 0 (bidirectional variant) */
  int zoh;     /* exact zero-order-hold input matrix instead of Δ·B */
  /* rows to compute: flat indices b*dim + d; NULL = all rows */
  const int64_t* rows;
  int64_t nrows;
  double* out;    /* [nrows, L] when rows != NULL, else [batch, dim, L] */
  double* h_last; /* [nrows, N] / [batch, dim, N]; may be NULL */
  /* work split */
  int64_t next_row;
  pthread_mutex_t lock;
} fwd_job;

/* The recurrence for one (b, d) row, sequential in t. */
static void scan_row(const fwd_job* j, int64_t b, int64_t d, double* out_row, double* hl_row) {
  const int64_t L = j->seqlen, N = j->dstate, Dm = j->dim;
  double h[64];
  for (int64_t n = 0; n < N; n++) {
    const int64_t s0 = (b * Dm + d) * N + n;
    h[n] = j->h0_f64 ? j->h0_f64[s0] : (j->h0 ? (double)j->h0[s0] : 0.0);
  }
  const double bias = j->delta_bias ? (double)j->delta_bias[d] : 0.0;
  const double Dd = j->D ? (double)j->D[d] : 0.0;
  for (int64_t s = 0; s < L; s++) {
    const int64_t t = j->reverse ? (L - 1 - s) : s;
    const int64_t e = (b * Dm + d) * L + t; /* element index into [B, D, L] */
    const double u = j->u_f64 ? j->u_f64[e] : load_in(j->u, e, j->in_dtype);
    const double x = load_in(j->delta, e, j->in_dtype) + bias;
    const double dt = j->delta_softplus ? softplus(x) : x;
    double y = 0.0;
    for (int64_t n = 0; n < N; n++) {
      const int64_t bc = (b * N + n) * L + t; /* index into [B, N, L] */
      const double Bv = load_in(j->B, bc, j->in_dtype);
      const double Cv = load_in(j->C, bc, j->in_dtype);
      const double a = (double)j->A[d * N + n];
      const double abar = exp(dt * a);     /* Ā = exp(Δ·A) */
      /* B̄ = Δ·B, or with zoh the exact zero-order hold (ΔA)^{-1}(exp(ΔA) - 1)·ΔB = (exp(ΔA) - 1)/A·B,
       * whose limit at A = 0 is Δ·B. */
      const double bbar = (j->zoh && a != 0.0) ? expm1(dt * a) / a : dt;
      h[n] = abar * h[n] + bbar * Bv * u;  /* h_t = Ā·h_{t-1} + B̄·u */
      y += Cv * h[n];                      /* C·h_t reads the updated state */
    }
    y += Dd * u;
    if (j->z) y *= silu(load_in(j->z, e, j->in_dtype));
    out_row[t] = y;
  }
  if (hl_row)
    for (int64_t n = 0; n < N; n++) hl_row[n] = h[n];
}

static void* fwd_worker(void* arg) {
  fwd_job* j = (fwd_job*)arg;
  const int64_t total = j->rows ? j->nrows : j->batch * j->dim;
  for (;;) {
    pthread_mutex_lock(&j->lock);
    const int64_t r = j->next_row++;
    pthread_mutex_unlock(&j->lock);
    if (r >= total) break;
    const int64_t flat = j->rows ? j->rows[r] : r;
    const int64_t b = flat / j->dim, d = flat % j->dim;
    scan_row(j, b, d, j->out + r * j->seqlen, j->h_last ? j->h_last + r * j->dstate : NULL);
  }
  return NULL;
}

/*
 * Selective-scan forward over every row (rows == NULL) or over the listed
 * rows only (flat b*dim + d indices; outputs are then packed per listed row).
 * nthreads <= 1 runs on the calling thread.  Returns 0, or -1 on bad sizes.
 */
int oracle_selscan_fwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int in_dtype,
                       const void* u, const void* delta, const float* A, const void* B, const void* C,
                       const float* D, const void* z, const float* delta_bias, int delta_softplus,
                       const float* h0, const double* h0_f64, int reverse, int zoh, const double* u_f64,
                       const int64_t* rows, int64_t nrows,
                       double* out,
                       double* h_last, int nthreads) {
  if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1 || dstate > 64) return -1;
  if (in_dtype != ORACLE_F32 && in_dtype != ORACLE_BF16) return -1;
  if ((!u && !u_f64) || !delta || !A || !B || !C || !out) return -1;
  fwd_job j;
  memset(&j, 0, sizeof j);
  j.batch = batch;
  j.dim = dim;
  j.seqlen = seqlen;
  j.dstate = dstate;
  j.in_dtype = in_dtype;
  j.u = u;
  j.delta = delta;
  j.z = z;
  j.B = B;
  j.C = C;
  j.A = A;
  j.D = D;
  j.delta_bias = delta_bias;
  j.h0 = h0;
  j.h0_f64 = h0_f64;
  j.delta_softplus = delta_softplus;
  j.reverse = reverse;
  j.zoh = zoh;
  j.u_f64 = u_f64;
  j.rows = rows;
  j.nrows = nrows;
  j.out = out;
  j.h_last = h_last;
  pthread_mutex_init(&j.lock, NULL);
  if (nthreads <= 1) {
    fwd_worker(&j);
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int i = 0; i < nthreads; i++)
      if (pthread_create(&th[i], NULL, fwd_worker, &j) == 0) started++;
      else break;
    if (started == 0) fwd_worker(&j);
    for (int i = 0; i < started; i++) pthread_join(th[i], NULL);
    free(th);
  }
  pthread_mutex_destroy(&j.lock);
  return 0;
}

/*
 * One recurrent decode step (the L = 1 case of the forward), in place on an
 * fp64 state [batch, dim, dstate]: the state after the step replaces it.
 * u, delta, z are [batch, dim]; B, C are [batch, dstate].
 * This is the constant-memory recurrent inference mode ("Mamba架构深度剖析" §3).
 */
int oracle_selscan_step(int64_t batch, int64_t dim, int64_t dstate, int in_dtype, const void* u,
                        const void* delta, const float* A, const void* B, const void* C, const float* D,
                        const void* z, const float* delta_bias, int delta_softplus, double* state,
                        double* out) {
  if (batch < 0 || dim < 0 || dstate < 1 || dstate > 64) return -1;
  if (!u || !delta || !A || !B || !C || !state || !out) return -1;
  for (int64_t b = 0; b < batch; b++) {
    for (int64_t d = 0; d < dim; d++) {
      const int64_t e = b * dim + d;
      const double uu = load_in(u, e, in_dtype);
      const double x = load_in(delta, e, in_dtype) + (delta_bias ? (double)delta_bias[d] : 0.0);
      const double dt = delta_softplus ? softplus(x) : x;
      double y = 0.0;
      for (int64_t n = 0; n < dstate; n++) {
        double* h = &state[e * dstate + n];
        const double Bv = load_in(B, b * dstate + n, in_dtype);
        const double Cv = load_in(C, b * dstate + n, in_dtype);
        *h = exp(dt * (double)A[d * dstate + n]) * (*h) + dt * Bv * uu;
        y += Cv * (*h);
      }
      y += (D ? (double)D[d] : 0.0) * uu;
      if (z) y *= silu(load_in(z, e, in_dtype));
      out[e] = y;
    }
  }
  return 0;
}

/*
 * Gradients of the forward (Δ·B discretisation, forward direction) for a loss whose gradient with
 * respect to out is dout [B, D, L] and with respect to h_last is dh_last [B, D, N] (NULL: zero).
 *
 * Reverse-mode differentiation of the recurrence above, taken in the reverse of the order it runs.
 * The forward of a row is first rerun keeping every state h_t (the pages' "recomputation": the
 * backward needs the states, which the forward does not store).  Then, with g the gradient with
 * respect to the state after the step being undone (starting from dh_last), for t = L-1 down to 0:
 *   y_t = Σ_n C_t[n] h_t[n] + D u_t,  out_t = y_t · silu(z_t)
 *     dy_t  = dout_t · silu(z_t)                      (dout_t without a gate)
 *     dz_t  = dout_t · y_t · silu'(z_t),  silu'(z) = σ(z)(1 + z(1 - σ(z)))
 *     dD   += dy_t · u_t,   du_t = dy_t · D
 *   for every state n, with G = g[n] + dy_t C_t[n] the full gradient with respect to h_t[n]:
 *     dC_t[n] += dy_t · h_t[n]
 *     h_t[n] = Ā_t[n] h_{t-1}[n] + Δ_t B_t[n] u_t, Ā_t[n] = exp(Δ_t A[n]):
 *       dB_t[n] += G Δ_t u_t,  du_t += G Δ_t B_t[n]
 *       dΔ_t    += G (B_t[n] u_t + A[n] Ā_t[n] h_{t-1}[n])
 *       dA[n]   += G Ā_t[n] h_{t-1}[n] Δ_t
 *       g[n]     = G Ā_t[n]                         (the gradient with respect to h_{t-1}[n])
 *   Δ_t = softplus(x_t), x_t = δ_t + Δ_bias:  dδ_t = dΔ_t σ(x_t) (dΔ_t without softplus), dΔ_bias += dδ_t
 * and finally dh0 = g.  B and C are shared by the channels of a batch entry and A, D, Δ_bias by the
 * batch entries of a channel, so their gradients are sums over those rows.
 *
 * Outputs are fp64: du, ddelta, dz [B, D, L] (dz may be NULL when z is), dA [D, N], dB, dC [B, N, L],
 * dD, dbias [D] (each may be NULL), dh0 [B, D, N] (may be NULL).  Sums over rows are formed per worker
 * thread (rows are dealt to workers in a fixed order) and added in worker order.
 */
typedef struct {
  int64_t batch, dim, seqlen, dstate;
  int in_dtype;
  const void *u, *delta, *z, *B, *C;
  const float *A, *D, *delta_bias, *h0;
  int delta_softplus;
  const double *dout, *dh_last;
  double *du, *ddelta, *dz, *dh0;
  int nthreads;
} bwd_job;

typedef struct {
  const bwd_job* j;
  int worker;
  double *dA, *dB, *dC, *dD, *dbias; /* this worker's partial sums */
  int failed;
} bwd_worker_t;

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

static void bwd_row(bwd_worker_t* w, int64_t b, int64_t d, double* hs, double* ys) {
  const bwd_job* j = w->j;
  const int64_t L = j->seqlen, N = j->dstate, Dm = j->dim;
  const double bias = j->delta_bias ? 1.0 * j->delta_bias[d] : 0.0;
  const double Dd = j->D ? 1.0 * j->D[d] : 0.0;
  /* Recomputation: hs[(t + 1) * N + n] = h_t[n] for t = -1 .. L-1, ys[t] = y_t. */
  for (int64_t n = 0; n < N; n++) hs[n] = j->h0 ? (double)j->h0[(b * Dm + d) * N + n] : 0.0;
  for (int64_t t = 0; t < L; t++) {
    const int64_t e = (b * Dm + d) * L + t;
    const double u = load_in(j->u, e, j->in_dtype);
    const double x = bias + load_in(j->delta, e, j->in_dtype);
    const double dt = j->delta_softplus ? softplus(x) : x;
    double y = Dd * u;
    for (int64_t n = 0; n < N; n++) {
      const int64_t bc = (b * N + n) * L + t;
      const double abar = exp(dt * (double)j->A[d * N + n]);
      const double h = abar * hs[t * N + n] + dt * load_in(j->B, bc, j->in_dtype) * u;
      hs[(t + 1) * N + n] = h;
      y += load_in(j->C, bc, j->in_dtype) * h;
    }
    ys[t] = y;
  }
  /* The reverse sweep. */
  double g[64];
  for (int64_t n = 0; n < N; n++) g[n] = j->dh_last ? j->dh_last[(b * Dm + d) * N + n] : 0.0;
  for (int64_t t = L - 1; t >= 0; t--) {
    const int64_t e = (b * Dm + d) * L + t;
    const double u = load_in(j->u, e, j->in_dtype);
    const double x = bias + load_in(j->delta, e, j->in_dtype);
    const double dt = j->delta_softplus ? softplus(x) : x;
    double dy = j->dout[e];
    if (j->z) {
      const double zz = load_in(j->z, e, j->in_dtype);
      const double sg = sigmoid(zz);
      if (j->dz) j->dz[e] = j->dout[e] * ys[t] * sg * (1.0 + zz * (1.0 - sg));
      dy = j->dout[e] * zz * sg;
    }
    if (w->dD) w->dD[d] += dy * u;
    double du = dy * Dd, ddt = 0.0;
    for (int64_t n = 0; n < N; n++) {
      const int64_t bc = (b * N + n) * L + t;
      const double Bv = load_in(j->B, bc, j->in_dtype), Cv = load_in(j->C, bc, j->in_dtype);
      const double a = j->A[d * N + n];
      const double abar = exp(a * dt); /* Ā_t[n] */
      const double hprev = hs[t * N + n];
      const double G = g[n] + dy * Cv;
      if (w->dC) w->dC[bc] += dy * hs[(t + 1) * N + n];
      if (w->dB) w->dB[bc] += G * dt * u;
      du += G * dt * Bv;
      ddt += G * (Bv * u + a * abar * hprev);
      if (w->dA) w->dA[d * N + n] += G * abar * hprev * dt;
      g[n] = G * abar;
    }
    const double dx = j->delta_softplus ? ddt * sigmoid(x) : ddt;
    j->du[e] = du;
    j->ddelta[e] = dx;
    if (w->dbias) w->dbias[d] += dx;
  }
  if (j->dh0)
    for (int64_t n = 0; n < N; n++) j->dh0[(b * Dm + d) * N + n] = g[n];
}

static void* bwd_worker(void* arg) {
  bwd_worker_t* w = (bwd_worker_t*)arg;
  const bwd_job* j = w->j;
  const int64_t L = j->seqlen, N = j->dstate;
  double* hs = (double*)malloc(sizeof(double) * (size_t)((L + 1) * N));
  double* ys = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
  if (!hs || !ys) {
    w->failed = 1;
  } else {
    for (int64_t r = w->worker; r < j->batch * j->dim; r += j->nthreads) bwd_row(w, r / j->dim, r % j->dim, hs, ys);
  }
  free(hs);
  free(ys);
  return NULL;
}

int oracle_selscan_bwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate, int in_dtype, const void* u,
                       const void* delta, const float* A, const void* B, const void* C, const float* D,
                       const void* z, const float* delta_bias, int delta_softplus, const float* h0,
                       const double* dout, const double* dh_last, double* du, double* ddelta, double* dz,
                       double* dA, double* dB, double* dC, double* dD, double* dbias, double* dh0, int nthreads) {
  if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1 || dstate > 64) return -1;
  if (in_dtype != ORACLE_F32 && in_dtype != ORACLE_BF16) return -1;
  if (!u || !delta || !A || !B || !C || !dout || !du || !ddelta) return -1;
  bwd_job j;
  memset(&j, 0, sizeof j);
  j.batch = batch;
  j.dim = dim;
  j.seqlen = seqlen;
  j.dstate = dstate;
  j.in_dtype = in_dtype;
  j.u = u;
  j.delta = delta;
  j.z = z;
  j.B = B;
  j.C = C;
  j.A = A;
  j.D = D;
  j.delta_bias = delta_bias;
  j.h0 = h0;
  j.delta_softplus = delta_softplus;
  j.dout = dout;
  j.dh_last = dh_last;
  j.du = du;
  j.ddelta = ddelta;
  j.dz = dz;
  j.dh0 = dh0;
  j.nthreads = nthreads > 1 ? nthreads : 1;
  const int nw = j.nthreads;
  const size_t nbc = (size_t)(batch * dstate * seqlen), na = (size_t)(dim * dstate), nd = (size_t)dim;
  bwd_worker_t* ws = (bwd_worker_t*)calloc((size_t)nw, sizeof(bwd_worker_t));
  if (!ws) return -2;
  int rc = 0;
  for (int k = 0; k < nw; k++) {
    ws[k].j = &j;
    ws[k].worker = k;
    ws[k].dA = dA ? (double*)calloc(na, sizeof(double)) : NULL;
    ws[k].dB = dB ? (double*)calloc(nbc ? nbc : 1, sizeof(double)) : NULL;
    ws[k].dC = dC ? (double*)calloc(nbc ? nbc : 1, sizeof(double)) : NULL;
    ws[k].dD = dD ? (double*)calloc(nd ? nd : 1, sizeof(double)) : NULL;
    ws[k].dbias = dbias ? (double*)calloc(nd ? nd : 1, sizeof(double)) : NULL;
    if ((dA && !ws[k].dA) || (dB && !ws[k].dB) || (dC && !ws[k].dC) || (dD && !ws[k].dD) || (dbias && !ws[k].dbias))
      rc = -2;
  }
  if (rc == 0) {
    if (nw == 1) {
      bwd_worker(&ws[0]);
    } else {
      pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nw);
      int started = 0;
      for (int k = 0; k < nw; k++)
        if (pthread_create(&th[k], NULL, bwd_worker, &ws[k]) == 0) started++;
        else break;
      for (int k = started; k < nw; k++) bwd_worker(&ws[k]); /* any worker that could not start runs here */
      for (int k = 0; k < started; k++) pthread_join(th[k], NULL);
      free(th);
    }
    if (dA) memset(dA, 0, na * sizeof(double));
    if (dB) memset(dB, 0, nbc * sizeof(double));
    if (dC) memset(dC, 0, nbc * sizeof(double));
    if (dD) memset(dD, 0, nd * sizeof(double));
    if (dbias) memset(dbias, 0, nd * sizeof(double));
    for (int k = 0; k < nw; k++) {
      if (ws[k].failed) rc = -2;
      for (size_t i = 0; dA && i < na; i++) dA[i] += ws[k].dA[i];
      for (size_t i = 0; dB && i < nbc; i++) dB[i] += ws[k].dB[i];
      for (size_t i = 0; dC && i < nbc; i++) dC[i] += ws[k].dC[i];
      for (size_t i = 0; dD && i < nd; i++) dD[i] += ws[k].dD[i];
      for (size_t i = 0; dbias && i < nd; i++) dbias[i] += ws[k].dbias[i];
    }
  }
  for (int k = 0; k < nw; k++) {
    free(ws[k].dA);
    free(ws[k].dB);
    free(ws[k].dC);
    free(ws[k].dD);
    free(ws[k].dbias);
  }
  free(ws);
  return rc;
}

/* Scalar helpers exposed for pinning the oracle's own building blocks. */
/*
 * The block's front before the scan: a causal depthwise 1-D convolution of width K over the
 * sequence, plus a per-channel bias, then SiLU ("Mamba架构与SSM模型：高效序列建模技术解析" §3.2:
 * d_conv = 4; "Mamba状态空间模型深度解析" §3.1: convolution then SiLU before the SSM):
 *   u[b,d,t] = silu( cb[d] + Σ_{k=0}^{K-1} w[d,k] · x[b,d,t-(K-1)+k] ),   x[.., t<0] = 0.
 * x is in_dtype [B, D, L]; w is fp32 [D, K]; cb is fp32 [D] or NULL.  Writes u in fp64.
 */
int oracle_conv_silu(int64_t batch, int64_t dim, int64_t seqlen, int64_t width, int in_dtype, const void* x,
                     const float* w, const float* cb, double* u_out) {
  if (batch < 0 || dim < 0 || seqlen < 0 || width < 1 || !x || !w || !u_out) return -1;
  for (int64_t b = 0; b < batch; b++)
    for (int64_t d = 0; d < dim; d++)
      for (int64_t t = 0; t < seqlen; t++) {
        double acc = cb ? (double)cb[d] : 0.0;
        for (int64_t k = 0; k < width; k++) {
          const int64_t tt = t - (width - 1) + k;
          if (tt >= 0) acc += (double)w[d * width + k] * load_in(x, (b * dim + d) * seqlen + tt, in_dtype);
        }
        u_out[(b * dim + d) * seqlen + t] = silu(acc);
      }
  return 0;
}

double oracle_softplus(double x) { return softplus(x); }
double oracle_silu(double z) { return silu(z); }
double oracle_load_bf16(uint16_t bits) { return load_in(&bits, 0, ORACLE_BF16); }
