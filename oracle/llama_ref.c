/*
 * Plain CPU oracle of one Llama-style decode step (test infrastructure only;
 * see llama_ref.h for the definitions followed and where they come from).
 *
 * Everything here is the plain definition written out: one loop per formula,
 * double precision, no blocking, fusion or reordering. The only concession to
 * speed is that the output rows of a matrix-vector product may be split over
 * threads; each row's dot product is still one sequential loop.
 */
#include "llama_ref.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16 <-> double                                                     */
/* ------------------------------------------------------------------ */

double ref_bf16_to_f64(uint16_t b) {
  /* a bf16 is the top half of an IEEE binary32 */
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

uint16_t ref_f64_to_bf16(double v) {
  float f = (float)v; /* round to nearest even, the kernels' activation precision */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) {
    return (uint16_t)((u >> 16) | 0x40u); /* keep NaN a NaN */
  }
  /* round the low 16 bits away, ties to even */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* single operations                                                   */
/* ------------------------------------------------------------------ */

void ref_rmsnorm(const double* x, const uint16_t* w, int n, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; ++i) out[i] = x[i] * inv * ref_bf16_to_f64(w[i]);
}

void ref_rope(double* v, int head_dim, int pos, double theta) {
  int half = head_dim / 2;
  for (int i = 0; i < half; ++i) {
    double freq = pow(theta, -2.0 * (double)i / (double)head_dim);
    double ang = (double)pos * freq;
    double c = cos(ang), s = sin(ang);
    double a = v[i], b = v[i + half];
    v[i] = a * c - b * s;
    v[i + half] = b * c + a * s;
  }
}

double ref_silu(double z) { return z / (1.0 + exp(-z)); }

typedef struct {
  const uint16_t* W;
  int cols;
  const double* x;
  double* y;
  int r0, r1;
} matvec_job;

static void* matvec_worker(void* arg) {
  matvec_job* j = (matvec_job*)arg;
  for (int r = j->r0; r < j->r1; ++r) {
    const uint16_t* row = j->W + (long)r * j->cols;
    double acc = 0.0;
    for (int c = 0; c < j->cols; ++c) acc += ref_bf16_to_f64(row[c]) * j->x[c];
    j->y[r] = acc;
  }
  return NULL;
}

void ref_matvec(const uint16_t* W, int rows, int cols, const double* x, double* y, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > rows) nthreads = rows > 0 ? rows : 1;
  matvec_job jobs[256];
  pthread_t tids[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].W = W;
    jobs[t].cols = cols;
    jobs[t].x = x;
    jobs[t].y = y;
    jobs[t].r0 = (int)((long)rows * t / nthreads);
    jobs[t].r1 = (int)((long)rows * (t + 1) / nthreads);
  }
  if (nthreads == 1) {
    matvec_worker(&jobs[0]);
    return;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&tids[t], NULL, matvec_worker, &jobs[t]);
  matvec_worker(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(tids[t], NULL);
}

void ref_attend(const double* q, const uint16_t* K, const uint16_t* V, int n, int head_dim,
                long stride, double scale, double* out) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double mx = -INFINITY;
  for (int t = 0; t < n; ++t) {
    double d = 0.0;
    for (int i = 0; i < head_dim; ++i) d += q[i] * ref_bf16_to_f64(K[(long)t * stride + i]);
    s[t] = d * scale;
    if (s[t] > mx) mx = s[t];
  }
  double den = 0.0;
  for (int t = 0; t < n; ++t) {
    s[t] = exp(s[t] - mx); /* the shift by the max cancels in the ratio */
    den += s[t];
  }
  for (int i = 0; i < head_dim; ++i) out[i] = 0.0;
  for (int t = 0; t < n; ++t) {
    double a = s[t] / den;
    for (int i = 0; i < head_dim; ++i) out[i] += a * ref_bf16_to_f64(V[(long)t * stride + i]);
  }
  free(s);
}

/* ------------------------------------------------------------------ */
/* whole decode step                                                   */
/* ------------------------------------------------------------------ */

static int config_ok(const ref_config* c) {
  if (!c) return 0;
  if (c->n_layers < 1 || c->hidden < 1 || c->n_heads < 1 || c->n_kv_heads < 1) return 0;
  if (c->head_dim < 2 || (c->head_dim & 1) || c->ffn < 1 || c->vocab < 1) return 0;
  if (c->n_heads % c->n_kv_heads) return 0;
  return 1;
}

int ref_decode_step(const ref_config* cfg, const ref_weights* w,
                    uint16_t* const* k_cache, uint16_t* const* v_cache,
                    int batch, int capacity,
                    const int32_t* tokens, const int32_t* positions,
                    double* logits_out, int nthreads) {
  if (!config_ok(cfg) || !w || !k_cache || !v_cache || !tokens || !positions || !logits_out)
    return -1;
  if (batch < 1 || capacity < 1) return -1;
  const int H = cfg->hidden, nh = cfg->n_heads, nkv = cfg->n_kv_heads, D = cfg->head_dim;
  const int F = cfg->ffn, V = cfg->vocab, L = cfg->n_layers;
  const int group = nh / nkv;
  for (int b = 0; b < batch; ++b) {
    if (tokens[b] < 0 || tokens[b] >= V) return -1;
    if (positions[b] < 0 || positions[b] >= capacity) return -1;
  }

  double* x = (double*)malloc(sizeof(double) * H);
  double* n = (double*)malloc(sizeof(double) * H);
  double* q = (double*)malloc(sizeof(double) * nh * D);
  double* k = (double*)malloc(sizeof(double) * nkv * D);
  double* v = (double*)malloc(sizeof(double) * nkv * D);
  double* att = (double*)malloc(sizeof(double) * nh * D);
  double* o = (double*)malloc(sizeof(double) * H);
  double* g = (double*)malloc(sizeof(double) * F);
  double* u = (double*)malloc(sizeof(double) * F);
  double* d = (double*)malloc(sizeof(double) * H);
  const double scale = 1.0 / sqrt((double)D);

  for (int b = 0; b < batch; ++b) {
    const int p = positions[b];
    /* embedding lookup */
    for (int i = 0; i < H; ++i) x[i] = ref_bf16_to_f64(w->embed[(long)tokens[b] * H + i]);

    for (int l = 0; l < L; ++l) {
      /* 1. RMSNorm + QKV + RoPE, then append k, v to the cache at slot p */
      ref_rmsnorm(x, w->attn_norm[l], H, cfg->rms_eps, n);
      ref_matvec(w->wq[l], nh * D, H, n, q, nthreads);
      ref_matvec(w->wk[l], nkv * D, H, n, k, nthreads);
      ref_matvec(w->wv[l], nkv * D, H, n, v, nthreads);
      for (int h = 0; h < nh; ++h) ref_rope(q + h * D, D, p, cfg->rope_theta);
      for (int h = 0; h < nkv; ++h) ref_rope(k + h * D, D, p, cfg->rope_theta);
      for (int h = 0; h < nkv; ++h) {
        long slot = (((long)b * nkv + h) * capacity + p) * D;
        for (int i = 0; i < D; ++i) {
          k_cache[l][slot + i] = ref_f64_to_bf16(k[h * D + i]);
          v_cache[l][slot + i] = ref_f64_to_bf16(v[h * D + i]);
        }
      }
      /* 2-3. attention of each q-head over slots 0..p of its kv-head */
      for (int h = 0; h < nh; ++h) {
        int kvh = h / group;
        long base = ((long)b * nkv + kvh) * capacity * D;
        ref_attend(q + h * D, k_cache[l] + base, v_cache[l] + base, p + 1, D, D, scale,
                   att + h * D);
      }
      /* 4. O-projection + residual */
      ref_matvec(w->wo[l], H, nh * D, att, o, nthreads);
      for (int i = 0; i < H; ++i) x[i] += o[i];
      /* 5. RMSNorm + up/gate + SiLU */
      ref_rmsnorm(x, w->mlp_norm[l], H, cfg->rms_eps, n);
      ref_matvec(w->wgate[l], F, H, n, g, nthreads);
      ref_matvec(w->wup[l], F, H, n, u, nthreads);
      for (int j = 0; j < F; ++j) g[j] = ref_silu(g[j]) * u[j];
      /* 6. down-projection + residual */
      ref_matvec(w->wdown[l], H, F, g, d, nthreads);
      for (int i = 0; i < H; ++i) x[i] += d[i];
    }
    /* 7. final RMSNorm + LM head */
    ref_rmsnorm(x, w->final_norm, H, cfg->rms_eps, n);
    const uint16_t* lm = cfg->tied ? w->embed : w->lm_head;
    ref_matvec(lm, V, H, n, logits_out + (long)b * V, nthreads);
  }

  free(x); free(n); free(q); free(k); free(v); free(att); free(o);
  free(g); free(u); free(d);
  return 0;
}

/* ------------------------------------------------------------------ */
/* full causal recompute (no cache)                                    */
/* ------------------------------------------------------------------ */

int ref_forward_full(const ref_config* cfg, const ref_weights* w, int nt,
                     const int32_t* tokens, double* logits_out,
                     uint16_t* const* k_out, uint16_t* const* v_out, int nthreads) {
  if (!config_ok(cfg) || !w || !tokens || !logits_out || nt < 1) return -1;
  const int H = cfg->hidden, nh = cfg->n_heads, nkv = cfg->n_kv_heads, D = cfg->head_dim;
  const int F = cfg->ffn, V = cfg->vocab, L = cfg->n_layers;
  const int group = nh / nkv;
  for (int t = 0; t < nt; ++t)
    if (tokens[t] < 0 || tokens[t] >= V) return -1;

  /* all n token rows at once, layer by layer */
  double* X = (double*)malloc(sizeof(double) * (size_t)nt * H);
  double* N = (double*)malloc(sizeof(double) * (size_t)nt * H);
  double* Q = (double*)malloc(sizeof(double) * (size_t)nt * nh * D);
  double* Kd = (double*)malloc(sizeof(double) * (size_t)nt * nkv * D);
  double* Vd = (double*)malloc(sizeof(double) * (size_t)nt * nkv * D);
  /* quantised K/V, laid out [nkv][n][D] so each head's keys are contiguous */
  uint16_t* Kq = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)nkv * nt * D);
  uint16_t* Vq = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)nkv * nt * D);
  double* A = (double*)malloc(sizeof(double) * (size_t)nt * nh * D);
  double* T = (double*)malloc(sizeof(double) * (size_t)nt * (F > H ? F : H));
  double* G = (double*)malloc(sizeof(double) * (size_t)nt * F);
  const double scale = 1.0 / sqrt((double)D);

  for (int t = 0; t < nt; ++t)
    for (int i = 0; i < H; ++i) X[(long)t * H + i] = ref_bf16_to_f64(w->embed[(long)tokens[t] * H + i]);

  for (int l = 0; l < L; ++l) {
    for (int t = 0; t < nt; ++t) {
      double* nrow = N + (long)t * H;
      ref_rmsnorm(X + (long)t * H, w->attn_norm[l], H, cfg->rms_eps, nrow);
      ref_matvec(w->wq[l], nh * D, H, nrow, Q + (long)t * nh * D, nthreads);
      ref_matvec(w->wk[l], nkv * D, H, nrow, Kd + (long)t * nkv * D, nthreads);
      ref_matvec(w->wv[l], nkv * D, H, nrow, Vd + (long)t * nkv * D, nthreads);
      for (int h = 0; h < nh; ++h) ref_rope(Q + ((long)t * nh + h) * D, D, t, cfg->rope_theta);
      for (int h = 0; h < nkv; ++h) ref_rope(Kd + ((long)t * nkv + h) * D, D, t, cfg->rope_theta);
      for (int h = 0; h < nkv; ++h)
        for (int i = 0; i < D; ++i) {
          Kq[((long)h * nt + t) * D + i] = ref_f64_to_bf16(Kd[((long)t * nkv + h) * D + i]);
          Vq[((long)h * nt + t) * D + i] = ref_f64_to_bf16(Vd[((long)t * nkv + h) * D + i]);
        }
    }
    if (k_out && k_out[l]) memcpy(k_out[l], Kq, sizeof(uint16_t) * (size_t)nkv * nt * D);
    if (v_out && v_out[l]) memcpy(v_out[l], Vq, sizeof(uint16_t) * (size_t)nkv * nt * D);
    /* causal attention: query row t sees key rows 0..t */
    for (int t = 0; t < nt; ++t)
      for (int h = 0; h < nh; ++h) {
        long base = (long)(h / group) * nt * D;
        ref_attend(Q + ((long)t * nh + h) * D, Kq + base, Vq + base, t + 1, D, D, scale,
                   A + ((long)t * nh + h) * D);
      }
    for (int t = 0; t < nt; ++t) {
      double* xrow = X + (long)t * H;
      double* trow = T + (long)t * H;
      ref_matvec(w->wo[l], H, nh * D, A + (long)t * nh * D, trow, nthreads);
      for (int i = 0; i < H; ++i) xrow[i] += trow[i];
    }
    for (int t = 0; t < nt; ++t) {
      double* nrow = N + (long)t * H;
      double* grow = G + (long)t * F;
      double* urow = T + (long)t * F;
      ref_rmsnorm(X + (long)t * H, w->mlp_norm[l], H, cfg->rms_eps, nrow);
      ref_matvec(w->wgate[l], F, H, nrow, grow, nthreads);
      ref_matvec(w->wup[l], F, H, nrow, urow, nthreads);
      for (int j = 0; j < F; ++j) grow[j] = ref_silu(grow[j]) * urow[j];
    }
    for (int t = 0; t < nt; ++t) {
      double* xrow = X + (long)t * H;
      double* trow = T + (long)t * H;
      ref_matvec(w->wdown[l], H, F, G + (long)t * F, trow, nthreads);
      for (int i = 0; i < H; ++i) xrow[i] += trow[i];
    }
  }
  const uint16_t* lm = cfg->tied ? w->embed : w->lm_head;
  for (int t = 0; t < nt; ++t) {
    ref_rmsnorm(X + (long)t * H, w->final_norm, H, cfg->rms_eps, N + (long)t * H);
    ref_matvec(lm, V, H, N + (long)t * H, logits_out + (long)t * V, nthreads);
  }
  free(X); free(N); free(Q); free(Kd); free(Vd); free(Kq); free(Vq);
  free(A); free(T); free(G);
  return 0;
}
