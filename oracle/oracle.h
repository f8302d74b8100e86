/*
 * oracle.h -- plain CPU reference of one low-batch transformer decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may load this library.  The
 * product path (decode_megakernel_sm_gb300) never links, imports or calls it.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes is the plain pre-norm decoder that the megakernel pages
 * describe as the work of one forward pass ("Megakernels: Deleting the Kernel
 * Boundary", section "Where the microseconds go": RMS norm, QKV projection,
 * RoPE, attention, output projection, residual add, norm, up and gate
 * projections, SiLU, down projection, residual, then the LM head), with the
 * opcode split of the same page's section "One launch, one interpreter".  The
 * MoE variant (router + top-k experts + shared MLP) follows "Gemma 4 TPU
 * megakernel", section "Megakernels for Gemma 4" (component table rows
 * Experts / Shared MLP / Router).
 *
 * Arithmetic: every value is a double; bf16 inputs are widened exactly.  The
 * only rounding the oracle does on purpose is the bf16 rounding (round to
 * nearest, ties to even, directly from double) of the K and V rows it appends
 * to the cache, because the cache is bf16, and, for int8 weights, the fp32
 * divisions that decide each code (orc_quantize_rows_int8).  No blocking,
 * fusion or reordering: dot products accumulate in index order.
 *
 * Pins (tests/test_oracle_pins.py): bf16 widening/rounding on printed bit
 * patterns, RMSNorm closed forms, RoPE identity at p=0 / norm preservation /
 * relative-position property / complex-rotation formulation, attention over
 * one position equals V and over equal scores equals mean(V), split-softmax
 * merge equals the unsplit softmax, GEMV against numpy float64 matmul,
 * SiLU closed forms, router top-k against a stable numpy argsort and E=1,k=1
 * MoE equal to the dense MLP, argmax first-index ties, and the whole tiny
 * decoder against an independent numpy formulation.  int8: worked rows of
 * the quantiser (ties to even, the clamp, a zero row), its half-step error
 * bound, the int8 GEMV against numpy on the dequantised matrix, and the
 * int8 decoder equal to the bf16 decoder on weights the quantiser
 * reproduces exactly.
 */
#ifndef MK_ORACLE_H
#define MK_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  double rms_eps, rope_theta;
  int n_experts, top_k, expert_ffn, shared_ffn; /* n_experts == 0: dense MLP */
  int max_seq;                                  /* cache rows per (b, kv head) */
} orc_config;

/* All weights are bf16 bit patterns in the usual [out][in] row-major layout.
 * Per-layer fields point at host arrays of n_layers pointers.             */
typedef struct {
  const uint16_t* embed;      /* [vocab][hidden] */
  const uint16_t* lm_head;    /* [vocab][hidden]; may equal embed (tied) */
  const uint16_t* final_norm; /* [hidden] */
  const uint16_t* const* attn_norm; /* [hidden] */
  const uint16_t* const* wq;        /* [n_q_heads*head_dim][hidden] */
  const uint16_t* const* wk;        /* [n_kv_heads*head_dim][hidden] */
  const uint16_t* const* wv;        /* [n_kv_heads*head_dim][hidden] */
  const uint16_t* const* wo;        /* [hidden][n_q_heads*head_dim] */
  const uint16_t* const* mlp_norm;  /* [hidden] */
  const uint16_t* const* w_gate;    /* dense: [ffn][hidden] */
  const uint16_t* const* w_up;      /* dense: [ffn][hidden] */
  const uint16_t* const* w_down;    /* dense: [hidden][ffn] */
  const uint16_t* const* router;    /* MoE: [n_experts][hidden] */
  const uint16_t* const* ex_gate;   /* MoE: [n_experts][expert_ffn][hidden] */
  const uint16_t* const* ex_up;     /* MoE: [n_experts][expert_ffn][hidden] */
  const uint16_t* const* ex_down;   /* MoE: [n_experts][hidden][expert_ffn] */
  const uint16_t* const* sh_gate;   /* MoE shared: [shared_ffn][hidden] */
  const uint16_t* const* sh_up;     /* MoE shared: [shared_ffn][hidden] */
  const uint16_t* const* sh_down;   /* MoE shared: [hidden][shared_ffn] */
  const struct orc_q8* q8;          /* NULL: bf16 weights; else int8 (below) */
} orc_weights;

/* int8 weights (the "INT8 experts" of "Gemma 4 TPU megakernel", section
 * "What's next", applied to every streamed matrix of a dense model): a
 * matrix is codes q[rows][cols] (int8) and one scale s[r] (fp32) per row,
 * standing for the weights w[r][k] = q[r][k] * s[r].                    */
typedef struct {
  const int8_t* codes;  /* [rows][cols] */
  const float* scales;  /* [rows] */
} orc_qmat;

/* With q8 set, orc_decode_step takes these matrices (per-layer arrays of
 * n_layers) in place of the bf16 wq, wk, wv, wo, w_gate, w_up, w_down and
 * lm_head; the embedding gather, norms and KV cache stay bf16.  Dense
 * models only.                                                           */
typedef struct orc_q8 {
  const orc_qmat* wq;
  const orc_qmat* wk;
  const orc_qmat* wv;
  const orc_qmat* wo;
  const orc_qmat* w_gate;
  const orc_qmat* w_up;
  const orc_qmat* w_down;
  orc_qmat lm_head;
} orc_q8;

/* bf16 <-> double */
double orc_bf16_to_f64(uint16_t h);
uint16_t orc_f64_to_bf16(double x);

/* out[i] = x[i] / sqrt(mean(x^2) + eps) * gain[i] */
void orc_rmsnorm(const double* x, const uint16_t* gain, int n, double eps, double* out);

/* Rotary embedding of one head vector v[d] at position pos, rotate-half
 * pairing (i, i + d/2) with frequency theta^(-2i/d). In place.          */
void orc_rope(double* v, int d, int pos, double theta);

/* y[r] = sum_k W[r][k] x[k] for a bf16 row-major W[rows][cols]. */
void orc_gemv(const uint16_t* W, int rows, int cols, const double* x, double* y);

/* Symmetric per-row int8 quantisation of a bf16 W[rows][cols]: with m the
 * largest |W[r][k]| of row r, s[r] = m / 127 and q[r][k] = W[r][k] / s[r]
 * rounded to the nearest integer, ties to even, then clamped to
 * [-127, 127]; both divisions are single-precision (fp32) and correctly
 * rounded, because the decision of an integer code is taken in the
 * precision the device takes it in.  A row of zeros: s = 0, codes 0.      */
void orc_quantize_rows_int8(const uint16_t* W, int rows, int cols, int8_t* codes, float* scales);

/* y[r] = sum_k (q[r][k] * s[r]) x[k]: the plain GEMV of the dequantised
 * weights (each q * s is exact in double).                                */
void orc_gemv_q8(const int8_t* codes, const float* scales, int rows, int cols, const double* x,
                 double* y);

/* Softmax attention of one query q[d] over n_pos cache rows K,V [n_pos][d]
 * (bf16), scale 1/sqrt(d).                                              */
void orc_attention(const double* q, const uint16_t* K, const uint16_t* V, int n_pos, int d,
                   double* out);

/* The same attention restricted to rows [p0, p1): returns the running max
 * m, the sum l of exp(s - m) and the unnormalised o = sum exp(s - m) V.
 * An empty range gives m = -inf, l = 0, o = 0.                          */
void orc_attention_partial(const double* q, const uint16_t* K, const uint16_t* V, int p0,
                           int p1, int d, double* m, double* l, double* o);

/* Combine n_parts partial states (m[n], l[n], o[n][d]) into the softmax
 * output out[d].                                                        */
void orc_attention_merge(int n_parts, const double* m, const double* l, const double* o, int d,
                         double* out);

double orc_silu(double a);

/* y = Wd (silu(Wg xn) * (Wu xn)) for Wg,Wu [F][H], Wd [H][F]; y is [H]. */
void orc_swiglu(const uint16_t* wg, const uint16_t* wu, const uint16_t* wd, int F, int H,
                const double* xn, double* y);

/* Softmax over E router logits, choose the k largest probabilities (ties:
 * lower expert id first), renormalise them to sum 1.  Writes ids[k], w[k]
 * and returns the relative margin (p_k - p_{k+1}) / p_k between the k-th
 * and (k+1)-th probability (1.0 when k == E).                           */
double orc_router_topk(const double* logits, int E, int k, int* ids, double* w);

/* First index of the maximum. */
int orc_argmax(const double* v, int n);

/* One decode step for B sequences.  tokens[b], positions[b] (P).  The new
 * K/V rows are rounded to bf16 and written at row P of kc[l] / vc[l], laid
 * out [B][n_kv_heads][max_seq][head_dim]; attention covers rows [0, P].
 * logits: [B][vocab], argmax: [B].
 * MoE only: route_ids [n_layers][B][top_k] and route_margin [n_layers][B]
 * receive the chosen experts and the top-k margin (may be NULL);
 * forced_routes (may be NULL) supplies expert ids per (layer, b) to use in
 * place of the oracle's own choice where forced_mask[layer*B+b] != 0.
 * Returns 0, or -1 on an invalid argument.                              */
int orc_decode_step(const orc_config* cfg, const orc_weights* w, uint16_t* const* kc,
                    uint16_t* const* vc, int B, const int* tokens, const int* positions,
                    double* logits, int* argmax, int* route_ids, double* route_margin,
                    const int* forced_routes, const int* forced_mask);

/* orc_decode_step that also records its intermediates (each may be NULL):
 * tq [n_layers][B][n_q_heads*head_dim] the queries after RoPE; tx
 * [2*n_layers][B][hidden] the residual after each O-projection (2l) and
 * after each MLP (2l+1); th [n_layers][B][ffn] SiLU(gate)*up (dense). The
 * arithmetic is that of orc_decode_step.                                  */
int orc_decode_step_trace(const orc_config* cfg, const orc_weights* w, uint16_t* const* kc,
                          uint16_t* const* vc, int B, const int* tokens, const int* positions,
                          double* logits, int* argmax, int* route_ids, double* route_margin,
                          const int* forced_routes, const int* forced_mask, double* tq,
                          double* tx, double* th);

/* orc_swiglu, also writing h = silu(Wg xn) * (Wu xn) when h != NULL. */
void orc_swiglu_h(const uint16_t* wg, const uint16_t* wu, const uint16_t* wd, int F, int H,
                  const double* xn, double* y, double* h);

void orc_set_threads(int n);
int orc_get_threads(void);

#ifdef __cplusplus
}
#endif
#endif
