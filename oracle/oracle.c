/*
 * Plain, slow, fp64 CPU oracle for the quantized sparse mixture-of-experts
 * FFN layer.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the CUDA library never does, and the
 * two share no code, header, table or helper.
 *
 * Sources (page title, then section):
 *  [P1] "Optimizing on-device inference for Apple Silicon" (Perplexity, 2026):
 *       "Qwen creates three distinct workload shapes" (router over 256 experts
 *       selecting eight, plus a shared expert that processes every token);
 *       "Dequantizing weights during matrix multiplication" (4-bit affine
 *       groups of 64 with a scale and a bias);  "Keeping expert routing on
 *       the GPU" (histogram, prefix scan, scatter, block map);  "Reducing
 *       intermediate and state traffic" (gate and up projections with their
 *       gated activation; expert output projection with its routing score
 *       and the shared expert's result).
 *  [P2] "Ember: packed Q8 decode" (voidwest.dev): the row-contiguous Q8_0
 *       source block, one fp16 scale and 32 int8 codes, 34 bytes.
 *  [P3] "oMLX MoE gate/up 融合优化：qwen35_moe_gate_up 实现剖析":
 *       "融合原理" (gate and up concatenated along the output axis, in
 *       [gate, up] order) and "前向传播补丁" (split, activation, then down).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - routing weights: softmax over the k selected logits (renormalize=1), or
 *    the full softmax over all E experts taken at the selected ones
 *    (renormalize=0);
 *  - top-k order: logit descending, ties to the lower expert index;
 *  - activation: silu(gate) * up with the gate half first;
 *  - the shared expert enters the sum with weight 1;
 *  - affine 4-bit: w = scale * q + bias, 8 codes per 32-bit word, lowest
 *    nibble first along the input axis;
 *  - grouping order inside an expert: stable by assignment id a = t*k + j.
 *
 * Everything is computed in double.  Inputs arrive as the raw bit patterns of
 * their storage types (bf16 and fp16 as uint16, fp32 as float), and are
 * decoded here from their IEEE / bfloat16 field definitions.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- numbers */

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 mantissa bits. */
double orc_bf16_to_f64(uint16_t b) {
  int sign = (b >> 15) & 1;
  int exp = (b >> 7) & 0xFF;
  int man = b & 0x7F;
  double v;
  if (exp == 0)
    v = ldexp((double)man, -126 - 7);          /* subnormal */
  else if (exp == 0xFF)
    v = man ? NAN : INFINITY;
  else
    v = ldexp(1.0 + (double)man / 128.0, exp - 127);
  return sign ? -v : v;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 mantissa bits. */
double orc_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int exp = (h >> 10) & 0x1F;
  int man = h & 0x3FF;
  double v;
  if (exp == 0)
    v = ldexp((double)man, -14 - 10);          /* subnormal */
  else if (exp == 0x1F)
    v = man ? NAN : INFINITY;
  else
    v = ldexp(1.0 + (double)man / 1024.0, exp - 15);
  return sign ? -v : v;
}

/* ------------------------------------------------------- quantized weights */

enum { ORC_Q8_0 = 0, ORC_AFFINE4_G64 = 1 };

/* One quantized weight tensor of shape [experts, rows, cols] (out, in).
 *  Q8_0 [P2]: codes int8 [experts, rows, cols]; one fp16 scale per 32
 *             consecutive inputs: scales [experts, rows, cols/32].
 *  AFFINE4_G64 [P1]: codes uint32 [experts, rows, cols/8], input c of a row in
 *             bits 4*(c%8) .. 4*(c%8)+3 of word c/8; one fp16 scale and one
 *             fp16 bias per 64 consecutive inputs: [experts, rows, cols/64]. */
typedef struct {
  int32_t qtype;
  int32_t experts, rows, cols;
  const void* codes;
  const uint16_t* scales;
  const uint16_t* biases;
} orc_qmat;

/* The real-valued weight W[e][n][c] that the stored bits represent. */
double orc_weight(const orc_qmat* m, int e, int n, int c) {
  size_t row = (size_t)e * m->rows + n;
  if (m->qtype == ORC_Q8_0) {
    const int8_t* q = (const int8_t*)m->codes;
    double code = (double)q[row * m->cols + c];
    double scale = orc_f16_to_f64(m->scales[row * (m->cols / 32) + c / 32]);
    return code * scale;
  } else {
    const uint32_t* w = (const uint32_t*)m->codes;
    uint32_t word = w[row * (m->cols / 8) + c / 8];
    double code = (double)((word >> (4 * (c % 8))) & 0xFu);
    double scale = orc_f16_to_f64(m->scales[row * (m->cols / 64) + c / 64]);
    double bias = orc_f16_to_f64(m->biases[row * (m->cols / 64) + c / 64]);
    return scale * code + bias;
  }
}

/* Storage size in bytes of one row of `cols` weights (codes plus per-group
 * metadata): 34 bytes per 32 for Q8_0 [P2], 4 bits per weight plus two fp16
 * per 64 for the affine format [P1]. */
int64_t orc_row_bytes(int32_t qtype, int32_t cols) {
  if (qtype == ORC_Q8_0) return (int64_t)(cols / 32) * (32 + 2);
  return (int64_t)(cols / 64) * (32 + 2 + 2);
}

/* y[n] = sum_c W[e][n][c] * x[c] for n < m->rows. */
void orc_qmatvec(const orc_qmat* m, int e, const double* x, double* y) {
  for (int n = 0; n < m->rows; ++n) {
    double acc = 0.0;
    for (int c = 0; c < m->cols; ++c) acc += orc_weight(m, e, n, c) * x[c];
    y[n] = acc;
  }
}

/* ----------------------------------------------------------------- router */

/* l[t][e] = sum_h x[t][h] * Wr[e][h] + bias[e]   [P1: the router scores each
 * of the experts for every token]. bias may be NULL. */
void orc_router_logits(const uint16_t* x_bf16, const float* w_router,
                       const float* bias, int32_t T, int32_t H, int32_t E,
                       double* logits) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += orc_bf16_to_f64(x_bf16[(size_t)t * H + h]) *
               (double)w_router[(size_t)e * H + h];
      if (bias) acc += (double)bias[e];
      logits[(size_t)t * E + e] = acc;
    }
  }
}

typedef struct {
  double v;
  int e;
} orc_scored;

static int orc_cmp_scored(const void* pa, const void* pb) {
  const orc_scored* a = (const orc_scored*)pa;
  const orc_scored* b = (const orc_scored*)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->e < b->e) ? -1 : (a->e > b->e);
}

/* Select the k experts of every token with the highest selection logits
 * sel (full sort descending, ties to the lower index), and their routing
 * weights from the weight logits wl:
 *   renormalize=1: w_j = exp(wl_j) / sum_{j'<k} exp(wl_j')  (softmax over
 *                  the selected experts);
 *   renormalize=0: w_j = exp(wl_j) / sum_{e<E} exp(wl_e).
 * sel == wl is the plain router [P1: the router scores the experts and keeps
 * eight].  sel = l + bias with wl = l is the selection-only bias variant: a
 * per-expert offset that changes which experts are chosen but not how their
 * outputs are weighted. */
void orc_topk_sel(const double* sel, const double* wl, int32_t T, int32_t E,
                  int32_t k, int32_t renormalize, int32_t* topk_idx,
                  double* topk_w) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    orc_scored* s = (orc_scored*)malloc(sizeof(orc_scored) * (size_t)E);
    for (int e = 0; e < E; ++e) {
      s[e].v = sel[(size_t)t * E + e];
      s[e].e = e;
    }
    qsort(s, (size_t)E, sizeof(orc_scored), orc_cmp_scored);
    const double* w = wl + (size_t)t * E;
    double top = w[s[0].e];
    if (renormalize) {
      for (int j = 1; j < k; ++j)
        if (w[s[j].e] > top) top = w[s[j].e];
    } else {
      for (int e = 1; e < E; ++e)
        if (w[e] > top) top = w[e];
    }
    double denom = 0.0;
    if (renormalize) {
      for (int j = 0; j < k; ++j) denom += exp(w[s[j].e] - top);
    } else {
      for (int e = 0; e < E; ++e) denom += exp(w[e] - top);
    }
    for (int j = 0; j < k; ++j) {
      topk_idx[(size_t)t * k + j] = s[j].e;
      topk_w[(size_t)t * k + j] = exp(w[s[j].e] - top) / denom;
    }
    free(s);
  }
}

/* The plain router: selection and weights from the same logits. */
void orc_topk(const double* logits, int32_t T, int32_t E, int32_t k,
              int32_t renormalize, int32_t* topk_idx, double* topk_w) {
  orc_topk_sel(logits, logits, T, E, k, renormalize, topk_idx, topk_w);
}

/* Shared-expert gate g[t] = 1 / (1 + exp(-sum_h x[t][h] * w_sg[h])), the
 * sigmoid of one more router-like row (reading of the shared-expert gate
 * variant: the pages run the shared expert on every token and name no gate;
 * this is its gated form). */
void orc_shared_gate(const uint16_t* x_bf16, const float* w_sg, int32_t T,
                     int32_t H, double* gate) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double z = 0.0;
    for (int h = 0; h < H; ++h)
      z += orc_bf16_to_f64(x_bf16[(size_t)t * H + h]) * (double)w_sg[h];
    gate[t] = 1.0 / (1.0 + exp(-z));
  }
}

/* --------------------------------------------------------------- grouping */

/* [P1 "Keeping expert routing on the GPU"]: a histogram counts the
 * assignments per expert, a prefix scan turns counts into start offsets, a
 * scatter places the rows into their expert groups, and a block map lists
 * the fixed-size blocks of rows the grouped matmul processes.
 *   assignment a = t*k + j goes to expert topk_idx[a];
 *   counts[e]     = #{a : topk_idx[a] == e};
 *   offsets[e]    = sum_{e'<e} counts[e'], offsets[E] = T*k;
 *   perm[i]       = the assignment at sorted position i, sorted by
 *                   (expert, a);  inv_perm[perm[i]] = i;
 *   tile_map      = pairs (e, offsets[e] + m*BM) for every expert e in
 *                   ascending order and m < ceil(counts[e]/BM);
 *   *n_tiles      = number of pairs.
 * Returns 0, or -1 if an expert id is out of range. */
int orc_group(const int32_t* topk_idx, int32_t T, int32_t k, int32_t E,
              int32_t BM, int32_t* counts, int32_t* offsets, int32_t* perm,
              int32_t* inv_perm, int32_t* tile_map, int32_t* n_tiles) {
  int64_t A = (int64_t)T * k;
  for (int64_t a = 0; a < A; ++a)
    if (topk_idx[a] < 0 || topk_idx[a] >= E) return -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t a = 0; a < A; ++a) counts[topk_idx[a]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int64_t pos = 0;
  for (int e = 0; e < E; ++e)
    for (int64_t a = 0; a < A; ++a)
      if (topk_idx[a] == e) perm[pos++] = (int32_t)a;
  for (int64_t i = 0; i < A; ++i) inv_perm[perm[i]] = (int32_t)i;
  int nt = 0;
  for (int e = 0; e < E; ++e)
    for (int m = 0; m * BM < counts[e]; ++m) {
      tile_map[2 * nt] = e;
      tile_map[2 * nt + 1] = offsets[e] + m * BM;
      ++nt;
    }
  *n_tiles = nt;
  return 0;
}

/* ------------------------------------------------------------- expert FFN */

/* silu(g) = g * sigmoid(g) = g / (1 + exp(-g)). */
double orc_silu(double g) { return g / (1.0 + exp(-g)); }

/* One expert applied to one token [P1 "Reducing intermediate and state
 * traffic", P3 "融合原理"]:
 *   gu = Wgu[e] x            (Wgu is [2I, H]: gate rows 0..I-1, up rows I..2I-1)
 *   h[i] = silu(gu[i]) * gu[I + i]
 *   o = Wdown[e] h           (Wdown is [H, I])
 * gu_out (2I) and h_out (I) may be NULL. */
void orc_expert_ffn(const orc_qmat* gate_up, const orc_qmat* down, int e,
                    const double* x, double* o, double* gu_out,
                    double* h_out) {
  int I = down->cols;
  double* gu = (double*)malloc(sizeof(double) * 2 * (size_t)I);
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  orc_qmatvec(gate_up, e, x, gu);
  for (int i = 0; i < I; ++i) h[i] = orc_silu(gu[i]) * gu[I + i];
  orc_qmatvec(down, e, h, o);
  if (gu_out) memcpy(gu_out, gu, sizeof(double) * 2 * (size_t)I);
  if (h_out) memcpy(h_out, h, sizeof(double) * (size_t)I);
  free(gu);
  free(h);
}

/* The layer output for the tokens listed in `tokens` (n_tok of them):
 *   y[t] = sum_{j<k} w[t][j] * o_{idx[t][j]}(x_t) + g[t] * o_shared(x_t)
 * with the routing (idx, w) given and g = shared_w (indexed by token), or
 * g = 1 when shared_w is NULL.  y is [n_tok, H], in the order of
 * `tokens`.  The k+1 expert outputs of a token are independent and are
 * computed in parallel; the sum is then taken in the order j = 0..k-1,
 * shared last. */
void orc_moe_layer_ex(const uint16_t* x_bf16, int32_t H, const int32_t* topk_idx,
                      const double* topk_w, int32_t k, const orc_qmat* gate_up,
                      const orc_qmat* down, const orc_qmat* shared_gate_up,
                      const orc_qmat* shared_down, const double* shared_w,
                      const int32_t* tokens, int32_t n_tok, double* y) {
  int64_t n_items = (int64_t)n_tok * (k + 1);
  double* o = (double*)malloc(sizeof(double) * (size_t)n_items * H);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t it = 0; it < n_items; ++it) {
    int64_t i = it / (k + 1);
    int j = (int)(it % (k + 1));
    int t = tokens[i];
    double* xt = (double*)malloc(sizeof(double) * (size_t)H);
    for (int c = 0; c < H; ++c)
      xt[c] = orc_bf16_to_f64(x_bf16[(size_t)t * H + c]);
    if (j < k)
      orc_expert_ffn(gate_up, down, topk_idx[(size_t)t * k + j], xt,
                     o + it * H, NULL, NULL);
    else
      orc_expert_ffn(shared_gate_up, shared_down, 0, xt, o + it * H, NULL,
                     NULL);
    free(xt);
  }
  for (int64_t i = 0; i < n_tok; ++i) {
    int t = tokens[i];
    for (int n = 0; n < H; ++n) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j)
        acc += topk_w[(size_t)t * k + j] * o[(i * (k + 1) + j) * H + n];
      acc += (shared_w ? shared_w[t] : 1.0) * o[(i * (k + 1) + k) * H + n];
      y[i * H + n] = acc;
    }
  }
  free(o);
}

/* The layer with the shared expert at weight 1. */
void orc_moe_layer(const uint16_t* x_bf16, int32_t H, const int32_t* topk_idx,
                   const double* topk_w, int32_t k, const orc_qmat* gate_up,
                   const orc_qmat* down, const orc_qmat* shared_gate_up,
                   const orc_qmat* shared_down, const int32_t* tokens,
                   int32_t n_tok, double* y) {
  orc_moe_layer_ex(x_bf16, H, topk_idx, topk_w, k, gate_up, down, shared_gate_up,
                   shared_down, NULL, tokens, n_tok, y);
}

/* ------------------------------------------------------------ dense GEMV */

/* y[n] = sum_c q[n][c] * d[n][c/32] * x[c]: one batch-1 Q8_0 projection
 * [P1 "Optimizing the single-row weight path"; P2 Q8_0 rows]. */
void orc_q8_gemv(const uint16_t* x_bf16, const int8_t* q, const uint16_t* d,
                 int32_t N, int32_t K, double* y) {
  double* x = (double*)malloc(sizeof(double) * (size_t)K);
  for (int c = 0; c < K; ++c) x[c] = orc_bf16_to_f64(x_bf16[c]);
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int c = 0; c < K; ++c)
      acc += (double)q[(size_t)n * K + c] *
             orc_f16_to_f64(d[(size_t)n * (K / 32) + c / 32]) * x[c];
    y[n] = acc;
  }
  free(x);
}

/* ----------------------------------------------------------------- misc */

/* ---------------------------------------- int8-activation Q8_0 GEMV mode */

/* Quantize the activation once into Q8_0-style blocks of 32 ("Ember: packed
 * Q8 decode": the Q/K/V and gate/up projections share one activation
 * quantization, and the dot products then run on 8-bit groups).  Reading
 * (the page gives no formula): per block b of 32 inputs, in fp32 as the
 * kernel computes it, d[b] = max|x| / 127 and q[i] = round-half-away(x[i] /
 * d[b]), clamped to [-127, 127]; an all-zero block has d = 0 and q = 0. */
void orc_q8_quantize_x(const uint16_t* x_bf16, int32_t K, int8_t* q, float* d) {
  for (int b = 0; b < K / 32; ++b) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
      const float v = (float)orc_bf16_to_f64(x_bf16[32 * b + i]);
      const float a = v < 0.0f ? -v : v;
      if (a > amax) amax = a;
    }
    const float db = amax / 127.0f;
    d[b] = db;
    for (int i = 0; i < 32; ++i) {
      float r = 0.0f;
      if (db != 0.0f) {
        const float v = (float)orc_bf16_to_f64(x_bf16[32 * b + i]);
        r = roundf(v / db);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
      }
      q[32 * b + i] = (int8_t)r;
    }
  }
}

/* y[n] = sum_b dw[n][b] * dx[b] * sum_{i in b} qw[n][i] * qx[i]: the Q8_0
 * GEMV on the quantized activation, each block's integer dot product exact,
 * the rest in double. */
void orc_q8_gemv_i8(const int8_t* qx, const float* dx, const int8_t* q,
                    const uint16_t* d, int32_t N, int32_t K, double* y) {
#pragma omp parallel for schedule(static)
  for (int n = 0; n < N; ++n) {
    double acc = 0.0;
    for (int b = 0; b < K / 32; ++b) {
      long long isum = 0;
      for (int i = 0; i < 32; ++i)
        isum += (long long)q[(size_t)n * K + 32 * b + i] * (long long)qx[32 * b + i];
      acc += orc_f16_to_f64(d[(size_t)n * (K / 32) + b]) * (double)dx[b] * (double)isum;
    }
    y[n] = acc;
  }
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
