/*
 * Plain CPU oracle of one Llama-style decode step (test infrastructure).
 *
 * This library exists only to check the CUDA decode path. Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path never does. It shares no code, header, table or constant with the CUDA
 * path.
 *
 * What it computes follows the seven fused instructions of the GPU interpreter
 * described on "3 · L'interpréteur sur GPU", §3.2 (table of the seven
 * instructions): RMSNorm + QKV + RoPE, attention, attention reduction,
 * O-projection + residual, RMSNorm + up/gate + SiLU, down-projection +
 * residual, RMSNorm + LM head. The pages name these operations but do not
 * define them, so the definitions used here are the textbook Llama ones:
 *
 *   RMSNorm(x, w)  = x / sqrt(mean(x^2) + eps) * w
 *   RoPE           rotate-half pairs (i, i + D/2), angle = pos * theta^(-2i/D)
 *   attention      softmax(q . k_t / sqrt(D)) over t = 0..pos (inclusive)
 *                  grouped-query: q-head h reads kv-head h / (nh / nkv)
 *   MLP            down( SiLU(gate(n)) * up(n) ),  SiLU(z) = z / (1 + e^-z)
 *
 * Precision: weights and the KV cache are bf16 (exactly widened to double);
 * every activation and accumulation is double. The new token's k and v are
 * quantised to bf16 before they are stored and read back, taking that decision
 * from the value rounded to fp32 (the precision the kernels keep activations
 * in), so both sides quantise from the same precision.
 *
 * Layouts: matrices are row-major [out][in] (the nn.Linear convention); the
 * KV cache of one layer is [batch][n_kv_heads][capacity][head_dim] bf16.
 *
 * What pins each function to something other than itself (the CPU tests
 * test_oracle_pins.py and test_oracle_model.py; "golden" is the file of
 * hand-derived values, each with its derivation):
 *   ref_bf16_to_f64 / ref_f64_to_bf16  exact widening of every bit pattern;
 *                     rounding against an independent library rounding;
 *                     golden rounding cases
 *   ref_rmsnorm       golden values; a constant vector's closed form; scale
 *                     invariance and unit RMS
 *   ref_rope          golden rotations; identity at position 0; pair norms
 *                     kept; scores that depend on the position difference
 *                     only; each pair's frequency theta^(-2i/D)
 *   ref_silu          golden values; its limits; SiLU(z) - SiLU(-z) = z
 *   ref_matvec        brute force on small matrices
 *   ref_attend        golden values; one key returns its value; equal keys
 *                     average the values; a library softmax;
 *                     split-and-combine equals one pass
 *   ref_decode_step   wiring cases with special weights (GQA map, attended
 *                     range, residual, MLP order, tied head, independent
 *                     batch rows); a whole step against the composition of
 *                     the pinned operations with nonzero q/k weights (a
 *                     planted wrong scale fails it)
 *   ref_forward_full  incremental decoding equals the full recompute
 */
#ifndef LLAMA_REF_H
#define LLAMA_REF_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int tied;            /* 1: the LM head is the embedding matrix */
  double rms_eps, rope_theta;
} ref_config;

/* bf16 bit patterns; per-layer arrays are host arrays of n_layers pointers */
typedef struct {
  const uint16_t* embed;       /* [V][H] */
  const uint16_t* lm_head;     /* [V][H]; ignored when tied */
  const uint16_t* final_norm;  /* [H] */
  const uint16_t* const* attn_norm; /* [H] */
  const uint16_t* const* wq;   /* [nh*D][H] */
  const uint16_t* const* wk;   /* [nkv*D][H] */
  const uint16_t* const* wv;   /* [nkv*D][H] */
  const uint16_t* const* wo;   /* [H][nh*D] */
  const uint16_t* const* mlp_norm; /* [H] */
  const uint16_t* const* wgate;    /* [F][H] */
  const uint16_t* const* wup;      /* [F][H] */
  const uint16_t* const* wdown;    /* [H][F] */
} ref_weights;

/* ---- scalar helpers -------------------------------------------------- */
double ref_bf16_to_f64(uint16_t b);
/* round to fp32 (nearest even), then to bf16 (nearest even) */
uint16_t ref_f64_to_bf16(double v);

/* ---- single operations (exported so the tests can pin each one) ------ */
void ref_rmsnorm(const double* x, const uint16_t* w, int n, double eps, double* out);
void ref_rope(double* v, int head_dim, int pos, double theta);
double ref_silu(double z);
/* y[r] = sum_c W[r][c] * x[c] for r < rows; W bf16 row-major [rows][cols] */
void ref_matvec(const uint16_t* W, int rows, int cols, const double* x, double* y, int nthreads);
/* one query head over n keys: out[D] = sum_t softmax_t(q.k_t * scale) v_t.
   K, V: bf16 rows of length head_dim with row stride `stride` elements. */
void ref_attend(const double* q, const uint16_t* K, const uint16_t* V, int n, int head_dim,
                long stride, double scale, double* out);

/* ---- whole decode step ----------------------------------------------- */
/* Decodes one token for each of `batch` sequences. Sequence b consumes
   tokens[b] at position positions[b]: its k/v are written into slot
   positions[b] of k_cache[l]/v_cache[l] and it attends to slots
   0..positions[b]. logits_out: [batch][V]. Returns 0, or -1 on invalid input. */
int ref_decode_step(const ref_config* cfg, const ref_weights* w,
                    uint16_t* const* k_cache, uint16_t* const* v_cache,
                    int batch, int capacity,
                    const int32_t* tokens, const int32_t* positions,
                    double* logits_out, int nthreads);

/* Full causal forward over n tokens of ONE sequence at positions 0..n-1, with
   no cache: every layer forms K and V for all n tokens at once (quantised to
   bf16 exactly as the cache is), and row i attends to rows 0..i.
   logits_out: [n][V]. Optionally returns the per-layer bf16 K/V rows in
   k_out[l]/v_out[l] ([nkv][n][D] each) when those pointers are non-NULL. */
int ref_forward_full(const ref_config* cfg, const ref_weights* w, int n,
                     const int32_t* tokens, double* logits_out,
                     uint16_t* const* k_out, uint16_t* const* v_out, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
