/*
 * gpt2_ref.c -- plain CPU oracle of one GPT-2 training step:
 * forward (with loss), zero_grad, backward, AdamW update.
 *
 * TEST INFRASTRUCTURE ONLY.  It is compiled and called by tests/, by
 * __graft_entry__.smoke() and by the CPU-baseline leg of bench.py; the CUDA
 * library never links, includes or calls it, and it shares no code with it.
 *
 * It is compiled twice: REAL=float (the fp32 reference the GPU path is
 * compared with) and REAL=double (finite-difference and library-routine
 * checks).  Every sum is accumulated in double and stored as REAL.  Loops are
 * the direct definitions; OpenMP only splits independent output elements, so
 * results do not depend on the thread count.
 *
 * Sources.  The llm.c web pages name the layers, the structs and the calls
 * of train_gpt2.c but print no formula and no code, so each routine below is
 * the textbook definition of the layer the pages name:
 *   [HX-1] page «llm.c：Andrej Karpathy带你从零复现LLM», section
 *          «核心代码解读：train_gpt2.c», item 1 (layer functions: encoder,
 *          layernorm, matmul, attention, gelu, residual, softmax,
 *          crossentropy, each forward and backward).
 *   [HX-2] same section, item 2 (ParameterTensors, ActivationTensors,
 *          GPT2Config, GPT2).
 *   [HX-3] same section, item 3 (gpt2_forward, gpt2_zero_grad,
 *          gpt2_backward, gpt2_update with AdamW).
 *   [QS]   page «千行C代码训完GPT-2» (新智元), section «快速入门»: the console
 *          log (num_parameters 124439808, num_activations 73323776 for
 *          B*T = 256) and Adam with learning rate 1e-4.
 *   [CU]   same page, section «纯CUDA也可训»: one preallocated 1-D buffer
 *          with every weight and activation pointing into it; the list of
 *          components (encoder, matmul, self-attention, GELU, residual,
 *          softmax, cross-entropy).
 *   [LL]   page «千行C代码训完GPT-2» (新智元): the plans for Llama2/Gemma-style
 *          models -- RMSNorm in place of layernorm, new layers such as RoPE.
 *          With cfg.llama set the model follows them: RMSNorm (no bias), RoPE
 *          on q and k (base 10000, interleaved pairs), no learned position
 *          table and no linear biases; the MLP stays GELU.
 * Readings where the pages are silent (GELU tanh form, layernorm eps 1e-5,
 * 1/sqrt(hs) attention scale, tied LM head without bias, (out,in) weight
 * orientation, padded vocab columns excluded from the softmax, AdamW with
 * bias correction and eps outside the square root) follow GPT-2 and PyTorch,
 * which the pages say llm.c matches exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef REAL
#define REAL float
#endif
typedef REAL real;

#define EXPORT __attribute__((visibility("default")))
#define LN_EPS 1e-5
#define GELU_C 0.044715

/* ======================================================================
 * Layer operations [HX-1].  Shapes: N rows (= B*T tokens), row-major.
 * Every *_backward ACCUMULATES (+=) into its gradient outputs.
 * ====================================================================== */

/* Token + position embedding [HX-1 encoder_forward]:
 *   x[b,t,:] = wte[ids[b,t],:] + wpe[t,:] */
EXPORT void encoder_forward(real* x, const int* ids, const real* wte, const real* wpe,
                            int B, int T, int C) {
  for (int b = 0; b < B; b++)
    for (int t = 0; t < T; t++) {
      const real* e = wte + (size_t)ids[b * T + t] * C;
      real* o = x + ((size_t)b * T + t) * C;
      if (wpe) {
        const real* p = wpe + (size_t)t * C;
        for (int c = 0; c < C; c++) o[c] = e[c] + p[c];
      } else {
        for (int c = 0; c < C; c++) o[c] = e[c];  /* no learned position table */
      }
    }
}

/* [HX-1 encoder_backward]: every position scatters its gradient row into the
 * wte row of its token and the wpe row of its position.  Contributions to one
 * destination row are summed in double in position order, then added once. */
EXPORT void encoder_backward(real* dwte, real* dwpe, const real* dx, const int* ids,
                             int B, int T, int C) {
  int N = B * T;
  double* acc = (double*)malloc(sizeof(double) * (size_t)C);
  for (int t = 0; t < T && dwpe; t++) {
    for (int c = 0; c < C; c++) acc[c] = 0.0;
    for (int b = 0; b < B; b++)
      for (int c = 0; c < C; c++) acc[c] += dx[((size_t)b * T + t) * C + c];
    for (int c = 0; c < C; c++) dwpe[(size_t)t * C + c] += (real)acc[c];
  }
  for (int p = 0; p < N; p++) {
    int id = ids[p], first = 1;
    for (int q = 0; q < p; q++)
      if (ids[q] == id) { first = 0; break; }
    if (!first) continue; /* this id was handled at its first position */
    for (int c = 0; c < C; c++) acc[c] = 0.0;
    for (int q = p; q < N; q++)
      if (ids[q] == id)
        for (int c = 0; c < C; c++) acc[c] += dx[(size_t)q * C + c];
    for (int c = 0; c < C; c++) dwte[(size_t)id * C + c] += (real)acc[c];
  }
  free(acc);
}

/* [HX-1 layernorm_forward]: per row, mean and biased variance over C,
 *   rstd = 1/sqrt(var + 1e-5),  y = (x - mean) * rstd * w + b. */
EXPORT void layernorm_forward(real* y, real* mean, real* rstd, const real* x,
                              const real* w, const real* bias, int N, int C) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < N; r++) {
    const real* xr = x + (size_t)r * C;
    double mu = 0.0, var = 0.0;
    for (int c = 0; c < C; c++) mu += xr[c];
    mu /= C;
    for (int c = 0; c < C; c++) var += (xr[c] - mu) * (xr[c] - mu);
    var /= C;
    double rs = 1.0 / sqrt(var + LN_EPS);
    for (int c = 0; c < C; c++)
      y[(size_t)r * C + c] = (real)((xr[c] - mu) * rs * w[c] + bias[c]);
    mean[r] = (real)mu;
    rstd[r] = (real)rs;
  }
}

/* [HX-1 layernorm_backward].  With n = (x - mean) * rstd and g = dy * w,
 * y = n*w + b gives
 *   dx = rstd * (g - mean_c(g) - n * mean_c(g * n)),
 *   dw = sum_rows dy * n,   db = sum_rows dy. */
EXPORT void layernorm_backward(real* dx, real* dw, real* db, const real* dy, const real* x,
                               const real* w, const real* mean, const real* rstd, int N, int C) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < N; r++) {
    const real* xr = x + (size_t)r * C;
    const real* dyr = dy + (size_t)r * C;
    double mu = mean[r], rs = rstd[r];
    double mg = 0.0, mgn = 0.0;
    for (int c = 0; c < C; c++) {
      double n = (xr[c] - mu) * rs, g = (double)dyr[c] * w[c];
      mg += g;
      mgn += g * n;
    }
    mg /= C;
    mgn /= C;
    for (int c = 0; c < C; c++) {
      double n = (xr[c] - mu) * rs, g = (double)dyr[c] * w[c];
      dx[(size_t)r * C + c] += (real)(rs * (g - mg - n * mgn));
    }
  }
#pragma omp parallel for schedule(static)
  for (int c = 0; c < C; c++) {
    double sw = 0.0, sb = 0.0;
    for (int r = 0; r < N; r++) {
      double n = (x[(size_t)r * C + c] - (double)mean[r]) * (double)rstd[r];
      sw += (double)dy[(size_t)r * C + c] * n;
      sb += dy[(size_t)r * C + c];
    }
    dw[c] += (real)sw;
    db[c] += (real)sb;
  }
}

/* [LL] RMSNorm: per row, rstd = 1/sqrt(mean_c(x^2) + 1e-5), y = x * rstd * w. */
EXPORT void rmsnorm_forward(real* y, real* rstd, const real* x, const real* w, int N, int C) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < N; r++) {
    const real* xr = x + (size_t)r * C;
    double ms = 0.0;
    for (int c = 0; c < C; c++) ms += (double)xr[c] * xr[c];
    ms /= C;
    double rs = 1.0 / sqrt(ms + LN_EPS);
    for (int c = 0; c < C; c++) y[(size_t)r * C + c] = (real)(xr[c] * rs * w[c]);
    rstd[r] = (real)rs;
  }
}

/* [LL] RMSNorm backward.  With n = x * rstd and g = dy * w, y = n*w gives
 *   dx = rstd * (g - n * mean_c(g * n)),   dw = sum_rows dy * n
 * (the layernorm formula without the mean(g) term: nothing is subtracted). */
EXPORT void rmsnorm_backward(real* dx, real* dw, const real* dy, const real* x, const real* w, const real* rstd,
                             int N, int C) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < N; r++) {
    const real* xr = x + (size_t)r * C;
    const real* dyr = dy + (size_t)r * C;
    double rs = rstd[r], mgn = 0.0;
    for (int c = 0; c < C; c++) mgn += (double)dyr[c] * w[c] * (xr[c] * rs);
    mgn /= C;
    for (int c = 0; c < C; c++) {
      double n = xr[c] * rs, g = (double)dyr[c] * w[c];
      dx[(size_t)r * C + c] += (real)(rs * (g - n * mgn));
    }
  }
  for (int c = 0; c < C; c++) {
    double a = 0.0;
    for (int r = 0; r < N; r++) a += (double)dy[(size_t)r * C + c] * (x[(size_t)r * C + c] * (double)rstd[r]);
    dw[c] += (real)a;
  }
}

/* [LL] rotary position embedding of q and k, in place in qkv (B,T,3C):
 * head h, pair i < hs/2 of token t is rotated by theta = t * 10000^(-2i/hs),
 *   (a, b) -> (a cos theta - b sin theta, a sin theta + b cos theta),
 * on the channels h*hs + 2i, h*hs + 2i + 1 of the q block and of the k block.
 * inverse != 0 rotates by -theta (the transpose: the backward of the map). */
EXPORT void rope_apply(real* qkv, int B, int T, int C, int NH, int inverse) {
  int hs = C / NH;
  for (int b = 0; b < B; b++)
    for (int t = 0; t < T; t++)
      for (int h = 0; h < NH; h++)
        for (int i = 0; i < hs / 2; i++) {
          double theta = t * pow(10000.0, -2.0 * i / hs);
          double cs = cos(theta), sn = inverse ? -sin(theta) : sin(theta);
          for (int part = 0; part < 2; part++) { /* q, then k */
            real* v = qkv + ((size_t)b * T + t) * 3 * C + part * C + h * hs + 2 * i;
            double a = v[0], bb = v[1];
            v[0] = (real)(a * cs - bb * sn);
            v[1] = (real)(a * sn + bb * cs);
          }
        }
}

/* [HX-1 matmul_forward]: out[r,o] = sum_i x[r,i] * W[o,i] + bias[o]
 * (W stored (OC, IC) row-major; bias may be NULL).  The sum over i runs in
 * index order for every output; W is read through a transposed copy only so
 * that consecutive outputs sit next to each other in memory. */
EXPORT void matmul_forward(real* out, const real* x, const real* W, const real* bias,
                           int N, int IC, int OC) {
  real* Wt = (real*)malloc(sizeof(real) * (size_t)IC * OC);
#pragma omp parallel for schedule(static)
  for (int i = 0; i < IC; i++)
    for (int o = 0; o < OC; o++) Wt[(size_t)i * OC + o] = W[(size_t)o * IC + i];
#pragma omp parallel
  {
    double* acc = (double*)malloc(sizeof(double) * (size_t)OC);
#pragma omp for schedule(static)
    for (int r = 0; r < N; r++) {
      for (int o = 0; o < OC; o++) acc[o] = 0.0;
      for (int i = 0; i < IC; i++) {
        double xi = x[(size_t)r * IC + i];
        const real* wr = Wt + (size_t)i * OC;
        for (int o = 0; o < OC; o++) acc[o] += xi * wr[o];
      }
      for (int o = 0; o < OC; o++)
        out[(size_t)r * OC + o] = (real)(acc[o] + (bias ? (double)bias[o] : 0.0));
    }
    free(acc);
  }
  free(Wt);
}

/* [HX-1 matmul_backward]: dx[r,i] += sum_o dy[r,o] W[o,i];
 * dW[o,i] += sum_r dy[r,o] x[r,i];  dbias[o] += sum_r dy[r,o]. */
EXPORT void matmul_backward(real* dx, real* dW, real* dbias, const real* dy, const real* x,
                            const real* W, int N, int IC, int OC) {
#pragma omp parallel
  {
    double* acc = (double*)malloc(sizeof(double) * (size_t)(IC > N ? IC : N));
#pragma omp for schedule(static)
    for (int r = 0; r < N; r++) {
      for (int i = 0; i < IC; i++) acc[i] = 0.0;
      for (int o = 0; o < OC; o++) {
        double g = dy[(size_t)r * OC + o];
        const real* wr = W + (size_t)o * IC;
        for (int i = 0; i < IC; i++) acc[i] += g * wr[i];
      }
      for (int i = 0; i < IC; i++) dx[(size_t)r * IC + i] += (real)acc[i];
    }
#pragma omp for schedule(static)
    for (int o = 0; o < OC; o++) {
      for (int i = 0; i < IC; i++) acc[i] = 0.0;
      double sb = 0.0;
      for (int r = 0; r < N; r++) {
        double g = dy[(size_t)r * OC + o];
        const real* xr = x + (size_t)r * IC;
        for (int i = 0; i < IC; i++) acc[i] += g * xr[i];
        sb += g;
      }
      for (int i = 0; i < IC; i++) dW[(size_t)o * IC + i] += (real)acc[i];
      if (dbias) dbias[o] += (real)sb;
    }
    free(acc);
  }
}

/* [HX-1 attention_forward], causal multi-head self-attention.
 * qkv is (B,T,3C): q = channels [0,C), k = [C,2C), v = [2C,3C); head h owns
 * channels [h*hs, (h+1)*hs) of each block, hs = C/NH.  For t2 <= t:
 *   preatt[t,t2] = q_t . k_t2 / sqrt(hs),  att = softmax over t2 <= t
 *   (max subtracted), out_t = sum_t2 att[t,t2] v_t2.
 * Masked entries (t2 > t) are stored as preatt = 0 and att = 0. */
EXPORT void attention_forward(real* out, real* preatt, real* att, const real* qkv,
                              int B, int T, int C, int NH) {
  int hs = C / NH;
  double scale = 1.0 / sqrt((double)hs);
#pragma omp parallel for collapse(3) schedule(static)
  for (int b = 0; b < B; b++)
    for (int h = 0; h < NH; h++)
      for (int t = 0; t < T; t++) {
        const real* q = qkv + ((size_t)b * T + t) * 3 * C + h * hs;
        real* pre = preatt + (((size_t)b * NH + h) * T + t) * T;
        real* a = att + (((size_t)b * NH + h) * T + t) * T;
        double mx = -INFINITY;
        for (int t2 = 0; t2 <= t; t2++) {
          const real* k = qkv + ((size_t)b * T + t2) * 3 * C + C + h * hs;
          double s = 0.0;
          for (int d = 0; d < hs; d++) s += (double)q[d] * k[d];
          s *= scale;
          pre[t2] = (real)s;
          if (s > mx) mx = s;
        }
        double sum = 0.0;
        for (int t2 = 0; t2 <= t; t2++) sum += exp((double)pre[t2] - mx);
        for (int t2 = 0; t2 < T; t2++) {
          if (t2 <= t) {
            a[t2] = (real)(exp((double)pre[t2] - mx) / sum);
          } else {
            a[t2] = 0;
            pre[t2] = 0;
          }
        }
        real* o = out + ((size_t)b * T + t) * C + h * hs;
        for (int d = 0; d < hs; d++) {
          double s = 0.0;
          for (int t2 = 0; t2 <= t; t2++)
            s += (double)a[t2] * qkv[((size_t)b * T + t2) * 3 * C + 2 * C + h * hs + d];
          o[d] = (real)s;
        }
      }
}

/* [HX-1 attention_backward], accumulating into dqkv.  With
 * da[t,t2] = dout_t . v_t2 (t2 <= t):
 *   dv_t2 += sum_t att[t,t2] dout_t
 *   ds[t,t2] = att[t,t2] (da[t,t2] - sum_j att[t,j] da[t,j])   (softmax)
 *   dq_t += sum_t2 ds[t,t2] k_t2 / sqrt(hs)
 *   dk_t2 += sum_t ds[t,t2] q_t / sqrt(hs) */
EXPORT void attention_backward(real* dqkv, const real* dout, const real* qkv, const real* att,
                               int B, int T, int C, int NH) {
  int hs = C / NH;
  double scale = 1.0 / sqrt((double)hs);
#pragma omp parallel for collapse(2) schedule(static)
  for (int b = 0; b < B; b++)
    for (int h = 0; h < NH; h++) {
      double* dq = (double*)calloc((size_t)T * hs, sizeof(double));
      double* dk = (double*)calloc((size_t)T * hs, sizeof(double));
      double* dv = (double*)calloc((size_t)T * hs, sizeof(double));
      double* da = (double*)malloc(sizeof(double) * (size_t)T);
      double* ds = (double*)malloc(sizeof(double) * (size_t)T);
      for (int t = 0; t < T; t++) {
        const real* a = att + (((size_t)b * NH + h) * T + t) * T;
        const real* go = dout + ((size_t)b * T + t) * C + h * hs;
        const real* q = qkv + ((size_t)b * T + t) * 3 * C + h * hs;
        double dot = 0.0;
        for (int t2 = 0; t2 <= t; t2++) {
          const real* v = qkv + ((size_t)b * T + t2) * 3 * C + 2 * C + h * hs;
          double s = 0.0;
          for (int d = 0; d < hs; d++) s += (double)go[d] * v[d];
          da[t2] = s;
          dot += (double)a[t2] * s;
          for (int d = 0; d < hs; d++) dv[(size_t)t2 * hs + d] += (double)a[t2] * go[d];
        }
        for (int t2 = 0; t2 <= t; t2++) ds[t2] = (double)a[t2] * (da[t2] - dot);
        for (int t2 = 0; t2 <= t; t2++) {
          const real* k = qkv + ((size_t)b * T + t2) * 3 * C + C + h * hs;
          for (int d = 0; d < hs; d++) {
            dq[(size_t)t * hs + d] += ds[t2] * k[d] * scale;
            dk[(size_t)t2 * hs + d] += ds[t2] * q[d] * scale;
          }
        }
      }
      for (int t = 0; t < T; t++)
        for (int d = 0; d < hs; d++) {
          real* row = dqkv + ((size_t)b * T + t) * 3 * C + h * hs + d;
          row[0] += (real)dq[(size_t)t * hs + d];
          row[C] += (real)dk[(size_t)t * hs + d];
          row[2 * C] += (real)dv[(size_t)t * hs + d];
        }
      free(dq); free(dk); free(dv); free(da); free(ds);
    }
}

/* [HX-1 gelu_forward], tanh form used by GPT-2:
 *   y = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
EXPORT void gelu_forward(real* y, const real* x, long long n) {
  double k = sqrt(2.0 / M_PI);
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < n; i++) {
    double v = x[i];
    y[i] = (real)(0.5 * v * (1.0 + tanh(k * (v + GELU_C * v * v * v))));
  }
}

/* [HX-1 gelu_backward]: with u = sqrt(2/pi) (x + 0.044715 x^3),
 *   dy/dx = 0.5 (1 + tanh u) + 0.5 x (1 - tanh^2 u) sqrt(2/pi) (1 + 3*0.044715 x^2) */
EXPORT void gelu_backward(real* dx, const real* x, const real* dy, long long n) {
  double k = sqrt(2.0 / M_PI);
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < n; i++) {
    double v = x[i];
    double th = tanh(k * (v + GELU_C * v * v * v));
    double d = 0.5 * (1.0 + th) + 0.5 * v * (1.0 - th * th) * k * (1.0 + 3.0 * GELU_C * v * v);
    dx[i] += (real)(d * dy[i]);
  }
}

/* [HX-1 residual_forward / residual_backward]: out = a + b; the gradient of
 * the sum flows unchanged to both summands. */
EXPORT void residual_forward(real* out, const real* a, const real* b, long long n) {
  for (long long i = 0; i < n; i++) out[i] = a[i] + b[i];
}
EXPORT void residual_backward(real* da, real* db, const real* dout, long long n) {
  for (long long i = 0; i < n; i++) {
    da[i] += dout[i];
    db[i] += dout[i];
  }
}

/* [HX-1 softmax_forward]: probs over the V real vocabulary columns of each
 * row (max subtracted); padded columns [V, Vp) get probability 0. */
EXPORT void softmax_forward(real* probs, const real* logits, int N, int V, int Vp) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < N; r++) {
    const real* l = logits + (size_t)r * Vp;
    real* p = probs + (size_t)r * Vp;
    double mx = -INFINITY, sum = 0.0;
    for (int v = 0; v < V; v++)
      if (l[v] > mx) mx = l[v];
    for (int v = 0; v < V; v++) sum += exp((double)l[v] - mx);
    for (int v = 0; v < V; v++) p[v] = (real)(exp((double)l[v] - mx) / sum);
    for (int v = V; v < Vp; v++) p[v] = 0;
  }
}

/* [HX-1 crossentropy_forward]: loss_r = -log probs[r, target_r]. */
EXPORT void crossentropy_forward(real* losses, const real* probs, const int* targets, int N, int Vp) {
  for (int r = 0; r < N; r++) losses[r] = (real)(-log((double)probs[(size_t)r * Vp + targets[r]]));
}

/* [HX-1 crossentropy_softmax_backward]: d loss_r / d logits[r,v]
 *   = dloss_r * (probs[r,v] - [v == target_r]) for v < V; padded columns
 * receive nothing. */
EXPORT void crossentropy_softmax_backward(real* dlogits, const real* dlosses, const real* probs,
                                          const int* targets, int N, int V, int Vp) {
#pragma omp parallel for schedule(static)
  for (int r = 0; r < N; r++)
    for (int v = 0; v < V; v++) {
      double ind = (v == targets[r]) ? 1.0 : 0.0;
      dlogits[(size_t)r * Vp + v] += (real)((double)dlosses[r] * ((double)probs[(size_t)r * Vp + v] - ind));
    }
}

/* [HX-3 gpt2_update] AdamW over n parameters, step t >= 1:
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2
 *   p -= lr * ( (m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps) + wd * p ) */
EXPORT void adamw_update(real* p, const real* g, real* m, real* v, long long n, double lr,
                         double b1, double b2, double eps, double wd, int t) {
  double c1 = 1.0 - pow(b1, t), c2 = 1.0 - pow(b2, t);
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < n; i++) {
    double gi = g[i];
    double mi = b1 * m[i] + (1.0 - b1) * gi;
    double vi = b2 * v[i] + (1.0 - b2) * gi * gi;
    double upd = (mi / c1) / (sqrt(vi / c2) + eps) + wd * p[i];
    m[i] = (real)mi;
    v[i] = (real)vi;
    p[i] = (real)(p[i] - lr * upd);
  }
}

/* ======================================================================
 * The model [HX-2]: GPT2Config, ParameterTensors (16 tensors in one flat
 * buffer), ActivationTensors (23 tensors in one flat buffer, [CU]).
 * ====================================================================== */

typedef struct {
  int max_seq_len, vocab_size, padded_vocab_size, num_layers, num_heads, channels;
  int llama; /* [LL]: RMSNorm, RoPE, no position table, no biases */
} ref_config;

enum {
  P_WTE, P_WPE, P_LN1W, P_LN1B, P_QKVW, P_QKVB, P_ATTPROJW, P_ATTPROJB,
  P_LN2W, P_LN2B, P_FCW, P_FCB, P_FCPROJW, P_FCPROJB, P_LNFW, P_LNFB, NUM_PARAM_TENSORS
};

enum {
  A_ENCODED, A_LN1, A_LN1_MEAN, A_LN1_RSTD, A_QKV, A_ATTY, A_PREATT, A_ATT, A_ATTPROJ,
  A_RESIDUAL2, A_LN2, A_LN2_MEAN, A_LN2_RSTD, A_FCH, A_FCH_GELU, A_FCPROJ, A_RESIDUAL3,
  A_LNF, A_LNF_MEAN, A_LNF_RSTD, A_LOGITS, A_PROBS, A_LOSSES, NUM_ACT_TENSORS
};

/* Element counts of the 16 parameter tensors; vocab_rows is V (the printed
 * count) or the padded Vp (the stored layout). */
static void param_sizes(const ref_config* c, long long vocab_rows, long long s[NUM_PARAM_TENSORS]) {
  long long L = c->num_layers, C = c->channels;
  s[P_WTE] = vocab_rows * C;
  s[P_WPE] = (long long)c->max_seq_len * C;
  s[P_LN1W] = L * C;
  s[P_LN1B] = L * C;
  s[P_QKVW] = L * 3 * C * C;
  s[P_QKVB] = L * 3 * C;
  s[P_ATTPROJW] = L * C * C;
  s[P_ATTPROJB] = L * C;
  s[P_LN2W] = L * C;
  s[P_LN2B] = L * C;
  s[P_FCW] = L * 4 * C * C;
  s[P_FCB] = L * 4 * C;
  s[P_FCPROJW] = L * C * 4 * C;
  s[P_FCPROJB] = L * C;
  s[P_LNFW] = C;
  s[P_LNFB] = C;
  if (c->llama) /* no position table, no biases (RMSNorm has no shift either) */
    s[P_WPE] = s[P_LN1B] = s[P_QKVB] = s[P_ATTPROJB] = s[P_LN2B] = s[P_FCB] = s[P_FCPROJB] = s[P_LNFB] = 0;
}

/* Element counts of the 23 activation tensors for a (B,T) batch; vocab_cols
 * is V (the printed count) or Vp (the stored layout). */
static void act_sizes(const ref_config* c, long long B, long long T, long long vocab_cols,
                      long long s[NUM_ACT_TENSORS]) {
  long long L = c->num_layers, C = c->channels, NH = c->num_heads, BT = B * T;
  s[A_ENCODED] = BT * C;
  s[A_LN1] = L * BT * C;
  s[A_LN1_MEAN] = L * BT;
  s[A_LN1_RSTD] = L * BT;
  s[A_QKV] = L * BT * 3 * C;
  s[A_ATTY] = L * BT * C;
  s[A_PREATT] = L * B * NH * T * T;
  s[A_ATT] = L * B * NH * T * T;
  s[A_ATTPROJ] = L * BT * C;
  s[A_RESIDUAL2] = L * BT * C;
  s[A_LN2] = L * BT * C;
  s[A_LN2_MEAN] = L * BT;
  s[A_LN2_RSTD] = L * BT;
  s[A_FCH] = L * BT * 4 * C;
  s[A_FCH_GELU] = L * BT * 4 * C;
  s[A_FCPROJ] = L * BT * C;
  s[A_RESIDUAL3] = L * BT * C;
  s[A_LNF] = BT * C;
  s[A_LNF_MEAN] = BT;
  s[A_LNF_RSTD] = BT;
  s[A_LOGITS] = BT * vocab_cols;
  s[A_PROBS] = BT * vocab_cols;
  s[A_LOSSES] = BT;
}

EXPORT long long ref_num_parameters(const ref_config* c, int padded) {
  long long s[NUM_PARAM_TENSORS], n = 0;
  param_sizes(c, padded ? c->padded_vocab_size : c->vocab_size, s);
  for (int i = 0; i < NUM_PARAM_TENSORS; i++) n += s[i];
  return n;
}

EXPORT long long ref_num_activations(const ref_config* c, int B, int T, int padded) {
  long long s[NUM_ACT_TENSORS], n = 0;
  act_sizes(c, B, T, padded ? c->padded_vocab_size : c->vocab_size, s);
  for (int i = 0; i < NUM_ACT_TENSORS; i++) n += s[i];
  return n;
}

/* Offset (elements) of parameter tensor `which` in the padded flat layout. */
EXPORT long long ref_param_offset(const ref_config* c, int which) {
  long long s[NUM_PARAM_TENSORS], off = 0;
  param_sizes(c, c->padded_vocab_size, s);
  for (int i = 0; i < which && i < NUM_PARAM_TENSORS; i++) off += s[i];
  return off;
}

typedef struct {
  ref_config cfg;
  int maxB, maxT;
  long long num_params;
  real *params, *grads, *m, *v;
  real *acts, *dacts;
  long long acts_capacity;
  real* P[NUM_PARAM_TENSORS];
  real* G[NUM_PARAM_TENSORS];
  real* A[NUM_ACT_TENSORS];
  real* dA[NUM_ACT_TENSORS];
  int* inputs;
  int* targets;
  int B, T, have_targets;
  double loss;
} ref_model;

static void carve(real* base, const long long* sizes, int n, real** out) {
  for (int i = 0; i < n; i++) {
    out[i] = base;
    base += sizes[i];
  }
}

EXPORT ref_model* ref_create(const ref_config* cfg, int maxB, int maxT) {
  ref_model* M = (ref_model*)calloc(1, sizeof(ref_model));
  if (!M) return NULL;
  M->cfg = *cfg;
  M->maxB = maxB;
  M->maxT = maxT;
  long long ps[NUM_PARAM_TENSORS];
  param_sizes(cfg, cfg->padded_vocab_size, ps);
  M->num_params = ref_num_parameters(cfg, 1);
  M->params = (real*)calloc((size_t)M->num_params, sizeof(real));
  M->grads = (real*)calloc((size_t)M->num_params, sizeof(real));
  M->m = (real*)calloc((size_t)M->num_params, sizeof(real));
  M->v = (real*)calloc((size_t)M->num_params, sizeof(real));
  M->acts_capacity = ref_num_activations(cfg, maxB, maxT, 1);
  M->acts = (real*)calloc((size_t)M->acts_capacity, sizeof(real));
  M->dacts = (real*)calloc((size_t)M->acts_capacity, sizeof(real));
  M->inputs = (int*)calloc((size_t)maxB * maxT, sizeof(int));
  M->targets = (int*)calloc((size_t)maxB * maxT, sizeof(int));
  if (!M->params || !M->grads || !M->m || !M->v || !M->acts || !M->dacts || !M->inputs || !M->targets) {
    free(M->params); free(M->grads); free(M->m); free(M->v);
    free(M->acts); free(M->dacts); free(M->inputs); free(M->targets); free(M);
    return NULL;
  }
  carve(M->params, ps, NUM_PARAM_TENSORS, M->P);
  carve(M->grads, ps, NUM_PARAM_TENSORS, M->G);
  return M;
}

EXPORT void ref_destroy(ref_model* M) {
  if (!M) return;
  free(M->params); free(M->grads); free(M->m); free(M->v);
  free(M->acts); free(M->dacts); free(M->inputs); free(M->targets);
  free(M);
}

EXPORT real* ref_params(ref_model* M) { return M->params; }
EXPORT real* ref_grads(ref_model* M) { return M->grads; }
EXPORT real* ref_m(ref_model* M) { return M->m; }
EXPORT real* ref_v(ref_model* M) { return M->v; }
EXPORT real* ref_act(ref_model* M, int which) { return M->A[which]; }
EXPORT long long ref_num_params_model(ref_model* M) { return M->num_params; }

/* [HX-3 gpt2_forward].  Returns the mean loss over B*T positions, or -1
 * when targets is NULL (logits only).  Returns -2 for a bad shape and -3 for
 * an out-of-range token id. */
EXPORT double ref_forward(ref_model* M, const int* inputs, const int* targets, int B, int T) {
  const ref_config* c = &M->cfg;
  int L = c->num_layers, C = c->channels, NH = c->num_heads;
  int V = c->vocab_size, Vp = c->padded_vocab_size;
  if (B < 1 || T < 1 || B > M->maxB || T > M->maxT || T > c->max_seq_len) return -2.0;
  int N = B * T;
  for (int i = 0; i < N; i++) {
    if (inputs[i] < 0 || inputs[i] >= V) return -3.0;
    if (targets && (targets[i] < 0 || targets[i] >= V)) return -3.0;
  }
  long long as[NUM_ACT_TENSORS];
  act_sizes(c, B, T, Vp, as);
  carve(M->acts, as, NUM_ACT_TENSORS, M->A);
  carve(M->dacts, as, NUM_ACT_TENSORS, M->dA);
  memcpy(M->inputs, inputs, sizeof(int) * (size_t)N);
  M->B = B;
  M->T = T;
  M->have_targets = targets != NULL;
  if (targets) memcpy(M->targets, targets, sizeof(int) * (size_t)N);

  real** P = M->P;
  real** A = M->A;
  size_t NC = (size_t)N * C, TT = (size_t)B * NH * T * T;
  const int ll = c->llama;
#define BIAS(t, off) (ll ? (const real*)NULL : P[t] + (off))
  encoder_forward(A[A_ENCODED], inputs, P[P_WTE], ll ? NULL : P[P_WPE], B, T, C);
  for (int l = 0; l < L; l++) {
    const real* x = l == 0 ? A[A_ENCODED] : A[A_RESIDUAL3] + (size_t)(l - 1) * NC;
    real* ln1 = A[A_LN1] + l * NC;
    real* qkv = A[A_QKV] + l * 3 * NC;
    real* atty = A[A_ATTY] + l * NC;
    real* preatt = A[A_PREATT] + l * TT;
    real* att = A[A_ATT] + l * TT;
    real* attproj = A[A_ATTPROJ] + l * NC;
    real* res2 = A[A_RESIDUAL2] + l * NC;
    real* ln2 = A[A_LN2] + l * NC;
    real* fch = A[A_FCH] + l * 4 * NC;
    real* fchg = A[A_FCH_GELU] + l * 4 * NC;
    real* fcproj = A[A_FCPROJ] + l * NC;
    real* res3 = A[A_RESIDUAL3] + l * NC;
    if (ll)
      rmsnorm_forward(ln1, A[A_LN1_RSTD] + (size_t)l * N, x, P[P_LN1W] + (size_t)l * C, N, C);
    else
      layernorm_forward(ln1, A[A_LN1_MEAN] + (size_t)l * N, A[A_LN1_RSTD] + (size_t)l * N, x,
                        P[P_LN1W] + (size_t)l * C, P[P_LN1B] + (size_t)l * C, N, C);
    matmul_forward(qkv, ln1, P[P_QKVW] + (size_t)l * 3 * C * C, BIAS(P_QKVB, (size_t)l * 3 * C), N, C, 3 * C);
    if (ll) rope_apply(qkv, B, T, C, NH, 0);
    attention_forward(atty, preatt, att, qkv, B, T, C, NH);
    matmul_forward(attproj, atty, P[P_ATTPROJW] + (size_t)l * C * C, BIAS(P_ATTPROJB, (size_t)l * C), N, C, C);
    residual_forward(res2, x, attproj, (long long)NC);
    if (ll)
      rmsnorm_forward(ln2, A[A_LN2_RSTD] + (size_t)l * N, res2, P[P_LN2W] + (size_t)l * C, N, C);
    else
      layernorm_forward(ln2, A[A_LN2_MEAN] + (size_t)l * N, A[A_LN2_RSTD] + (size_t)l * N, res2,
                        P[P_LN2W] + (size_t)l * C, P[P_LN2B] + (size_t)l * C, N, C);
    matmul_forward(fch, ln2, P[P_FCW] + (size_t)l * 4 * C * C, BIAS(P_FCB, (size_t)l * 4 * C), N, C, 4 * C);
    gelu_forward(fchg, fch, (long long)(4 * NC));
    matmul_forward(fcproj, fchg, P[P_FCPROJW] + (size_t)l * 4 * C * C, BIAS(P_FCPROJB, (size_t)l * C), N, 4 * C, C);
    residual_forward(res3, res2, fcproj, (long long)NC);
  }
  if (ll)
    rmsnorm_forward(A[A_LNF], A[A_LNF_RSTD], A[A_RESIDUAL3] + (size_t)(L - 1) * NC, P[P_LNFW], N, C);
  else
    layernorm_forward(A[A_LNF], A[A_LNF_MEAN], A[A_LNF_RSTD], A[A_RESIDUAL3] + (size_t)(L - 1) * NC,
                      P[P_LNFW], P[P_LNFB], N, C);
#undef BIAS
  /* LM head tied to wte, no bias; all Vp columns are computed. */
  matmul_forward(A[A_LOGITS], A[A_LNF], P[P_WTE], NULL, N, C, Vp);
  softmax_forward(A[A_PROBS], A[A_LOGITS], N, V, Vp);
  if (!targets) {
    M->loss = -1.0;
    return -1.0;
  }
  crossentropy_forward(A[A_LOSSES], A[A_PROBS], targets, N, Vp);
  double s = 0.0;
  for (int i = 0; i < N; i++) s += A[A_LOSSES][i];
  M->loss = s / N;
  return M->loss;
}

/* [HX-3 gpt2_zero_grad]: zero the parameter gradients and the activation
 * gradients. */
EXPORT void ref_zero_grad(ref_model* M) {
  memset(M->grads, 0, sizeof(real) * (size_t)M->num_params);
  memset(M->dacts, 0, sizeof(real) * (size_t)M->acts_capacity);
}

/* [HX-3 gpt2_backward]: accumulates the gradient of the mean loss into the
 * parameter gradients.  Activation gradients are scratch and are cleared
 * first, so two calls without zero_grad double the parameter gradients.
 * Returns -4 without a preceding forward that had targets. */
EXPORT int ref_backward(ref_model* M) {
  if (!M->have_targets) return -4;
  const ref_config* c = &M->cfg;
  int L = c->num_layers, C = c->channels, NH = c->num_heads;
  int V = c->vocab_size, Vp = c->padded_vocab_size;
  int B = M->B, T = M->T, N = B * T;
  size_t NC = (size_t)N * C;
  real** P = M->P;
  real** G = M->G;
  real** A = M->A;
  real** dA = M->dA;
  memset(M->dacts, 0, sizeof(real) * (size_t)ref_num_activations(c, B, T, 1));

  /* the mean over N positions: dloss_r = 1/N */
  for (int i = 0; i < N; i++) dA[A_LOSSES][i] = (real)(1.0 / N);
  crossentropy_softmax_backward(dA[A_LOGITS], dA[A_LOSSES], A[A_PROBS], M->targets, N, V, Vp);
  matmul_backward(dA[A_LNF], G[P_WTE], NULL, dA[A_LOGITS], A[A_LNF], P[P_WTE], N, C, Vp);
  real* resL = A[A_RESIDUAL3] + (size_t)(L - 1) * NC;
  real* dresL = dA[A_RESIDUAL3] + (size_t)(L - 1) * NC;
  const int ll = c->llama;
#define DBIAS(t, off) (ll ? (real*)NULL : G[t] + (off))
  if (ll)
    rmsnorm_backward(dresL, G[P_LNFW], dA[A_LNF], resL, P[P_LNFW], A[A_LNF_RSTD], N, C);
  else
    layernorm_backward(dresL, G[P_LNFW], G[P_LNFB], dA[A_LNF], resL, P[P_LNFW], A[A_LNF_MEAN],
                       A[A_LNF_RSTD], N, C);
  for (int l = L - 1; l >= 0; l--) {
    const real* x = l == 0 ? A[A_ENCODED] : A[A_RESIDUAL3] + (size_t)(l - 1) * NC;
    real* dx = l == 0 ? dA[A_ENCODED] : dA[A_RESIDUAL3] + (size_t)(l - 1) * NC;
    size_t TT = (size_t)B * NH * T * T;
    real* dres3 = dA[A_RESIDUAL3] + l * NC;
    real* dres2 = dA[A_RESIDUAL2] + l * NC;
    /* res3 = res2 + fcproj */
    residual_backward(dres2, dA[A_FCPROJ] + l * NC, dres3, (long long)NC);
    matmul_backward(dA[A_FCH_GELU] + l * 4 * NC, G[P_FCPROJW] + (size_t)l * 4 * C * C,
                    DBIAS(P_FCPROJB, (size_t)l * C), dA[A_FCPROJ] + l * NC, A[A_FCH_GELU] + l * 4 * NC,
                    P[P_FCPROJW] + (size_t)l * 4 * C * C, N, 4 * C, C);
    gelu_backward(dA[A_FCH] + l * 4 * NC, A[A_FCH] + l * 4 * NC, dA[A_FCH_GELU] + l * 4 * NC,
                  (long long)(4 * NC));
    matmul_backward(dA[A_LN2] + l * NC, G[P_FCW] + (size_t)l * 4 * C * C, DBIAS(P_FCB, (size_t)l * 4 * C),
                    dA[A_FCH] + l * 4 * NC, A[A_LN2] + l * NC, P[P_FCW] + (size_t)l * 4 * C * C, N, C, 4 * C);
    if (ll)
      rmsnorm_backward(dres2, G[P_LN2W] + (size_t)l * C, dA[A_LN2] + l * NC, A[A_RESIDUAL2] + l * NC,
                       P[P_LN2W] + (size_t)l * C, A[A_LN2_RSTD] + (size_t)l * N, N, C);
    else
      layernorm_backward(dres2, G[P_LN2W] + (size_t)l * C, G[P_LN2B] + (size_t)l * C, dA[A_LN2] + l * NC,
                         A[A_RESIDUAL2] + l * NC, P[P_LN2W] + (size_t)l * C, A[A_LN2_MEAN] + (size_t)l * N,
                         A[A_LN2_RSTD] + (size_t)l * N, N, C);
    /* res2 = x + attproj */
    residual_backward(dx, dA[A_ATTPROJ] + l * NC, dres2, (long long)NC);
    matmul_backward(dA[A_ATTY] + l * NC, G[P_ATTPROJW] + (size_t)l * C * C, DBIAS(P_ATTPROJB, (size_t)l * C),
                    dA[A_ATTPROJ] + l * NC, A[A_ATTY] + l * NC, P[P_ATTPROJW] + (size_t)l * C * C, N, C, C);
    attention_backward(dA[A_QKV] + l * 3 * NC, dA[A_ATTY] + l * NC, A[A_QKV] + l * 3 * NC,
                       A[A_ATT] + l * TT, B, T, C, NH);
    /* q and k were rotated after the matmul: carry their gradients back through the rotation */
    if (ll) rope_apply(dA[A_QKV] + l * 3 * NC, B, T, C, NH, 1);
    matmul_backward(dA[A_LN1] + l * NC, G[P_QKVW] + (size_t)l * 3 * C * C, DBIAS(P_QKVB, (size_t)l * 3 * C),
                    dA[A_QKV] + l * 3 * NC, A[A_LN1] + l * NC, P[P_QKVW] + (size_t)l * 3 * C * C, N, C, 3 * C);
    if (ll)
      rmsnorm_backward(dx, G[P_LN1W] + (size_t)l * C, dA[A_LN1] + l * NC, x, P[P_LN1W] + (size_t)l * C,
                       A[A_LN1_RSTD] + (size_t)l * N, N, C);
    else
      layernorm_backward(dx, G[P_LN1W] + (size_t)l * C, G[P_LN1B] + (size_t)l * C, dA[A_LN1] + l * NC, x,
                         P[P_LN1W] + (size_t)l * C, A[A_LN1_MEAN] + (size_t)l * N, A[A_LN1_RSTD] + (size_t)l * N,
                         N, C);
  }
#undef DBIAS
  encoder_backward(G[P_WTE], ll ? NULL : G[P_WPE], dA[A_ENCODED], M->inputs, B, T, C);
  return 0;
}

/* [HX-3 gpt2_update]: AdamW over the whole flat parameter buffer. */
EXPORT void ref_update(ref_model* M, double lr, double b1, double b2, double eps, double wd, int t) {
  adamw_update(M->params, M->grads, M->m, M->v, M->num_params, lr, b1, b2, eps, wd, t);
}
