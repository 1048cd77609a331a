/*
 * oracle.c -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * Plain fp64 CPU statement of one decode step (see oracle.h for the scope,
 * the sources and the two roundings that belong to the definition).  Every
 * function is written straight from its definition: no blocking, no fusion,
 * sums in index order.  OpenMP only splits independent output rows across
 * threads; it does not change any sum.
 *
 * Sources cited below:
 *   [Cohere]    "Cohere: a decode megakernel for North Mini Code" (the English
 *               and the Chinese text of the same article).
 *   [tiny-vllm] "tiny-vllm 5. The decode path that produces one token".
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "../synth/synth.h"

/* ---------------------------------------------------------------- helpers */

void orc_dense_row(const void* ctx, int row, double* out) {
  const orc_dense* m = (const orc_dense*)ctx;
  memcpy(out, m->data + (size_t)row * (size_t)m->cols, sizeof(double) * (size_t)m->cols);
}

static double dot(int n, const double* a, const double* b) {
  double s = 0.0;
  for (int i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

/* ---------------------------------------------------- layer operations */

/* RMSNorm: out_i = x_i / sqrt(mean_j x_j^2 + eps) * gamma_i.
 * [Cohere] "1. Reduce wave quantization": attention and the MoE read the same
 * normalized input; the layer ends in a fused residual add + RMSNorm. */
void orc_rmsnorm(int n, const double* x, const double* gamma, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += x[i] * x[i];
  const double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; ++i) out[i] = x[i] * inv * (gamma ? gamma[i] : 1.0);
}

/* RoPE on one head vector, in place: the pair (2i, 2i+1) is rotated by the
 * angle pos * theta_i, theta_i = base^(-2i/d), with no frequency scaling.
 * [tiny-vllm] "RoPE: one current position, recomputed on every call". */
void orc_rope(int d, double* v, int64_t pos, double base) {
  for (int i = 0; i < d / 2; ++i) {
    const double theta = pow(base, -(double)(2 * i) / (double)d);
    const double a = (double)pos * theta;
    const double c = cos(a), s = sin(a);
    const double x0 = v[2 * i], x1 = v[2 * i + 1];
    v[2 * i] = x0 * c - x1 * s;
    v[2 * i + 1] = x0 * s + x1 * c;
  }
}

/* softmax(s)_i = exp(s_i - max s) / sum_j exp(s_j - max s). */
void orc_softmax(int n, const double* s, double* p) {
  double mx = -INFINITY;
  for (int i = 0; i < n; ++i) mx = s[i] > mx ? s[i] : mx;
  double z = 0.0;
  for (int i = 0; i < n; ++i) {
    p[i] = exp(s[i] - mx);
    z += p[i];
  }
  for (int i = 0; i < n; ++i) p[i] /= z;
}

/* SiLU(x) = x / (1 + exp(-x)).  [Cohere] "Tasks": the expert up/gate GEMM
 * fuses the SiLU-and-multiply in its epilogue. */
double orc_silu(double x) { return x / (1.0 + exp(-x)); }

/* y = W x for W given row by row ([Cohere] "Tasks": every projection of the
 * decode step is a matrix-vector product at batch 1). */
void orc_matvec(const orc_matrix* W, const double* x, double* y) {
#pragma omp parallel
  {
    double* row = (double*)malloc(sizeof(double) * (size_t)W->cols);
#pragma omp for schedule(static)
    for (int r = 0; r < W->rows; ++r) {
      W->row(W->ctx, r, row);
      y[r] = dot(W->cols, row, x);
    }
    free(row);
  }
}

/* Softmax attention of one query over n keys: out = sum_t p_t V_t with
 * p = softmax(scale * q.K_t).  [Cohere] "Tasks": attention of the new token
 * over its KV; [tiny-vllm] "Attention is finished off by
 * pagedAttentionKernel": iterating only up to the sequence length is the mask. */
void orc_attend(int d, int n, const double* q, const double* K, const double* V, double scale,
                double* out) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double* p = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int t = 0; t < n; ++t) s[t] = scale * dot(d, q, K + (size_t)t * d);
  orc_softmax(n, s, p);
  for (int i = 0; i < d; ++i) {
    double acc = 0.0;
    for (int t = 0; t < n; ++t) acc += p[t] * V[(size_t)t * d + i];
    out[i] = acc;
  }
  free(s);
  free(p);
}

/* Attention over one KV slice, left unnormalised: m = max_t s_t,
 * l = sum_t exp(s_t - m), o = sum_t exp(s_t - m) V_t.  [Cohere] "Tasks":
 * ATTN_DECODE computes attention on a partial KV slice.  An empty slice gives
 * m = -inf, l = 0, o = 0. */
void orc_attend_partial(int d, int n, const double* q, const double* K, const double* V,
                        double scale, double* m, double* l, double* o) {
  double mx = -INFINITY;
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (int t = 0; t < n; ++t) {
    s[t] = scale * dot(d, q, K + (size_t)t * d);
    mx = s[t] > mx ? s[t] : mx;
  }
  double z = 0.0;
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  for (int t = 0; t < n; ++t) {
    const double e = exp(s[t] - mx);
    z += e;
    for (int i = 0; i < d; ++i) o[i] += e * V[(size_t)t * d + i];
  }
  *m = mx;
  *l = z;
  free(s);
}

/* Merge of slice partials into the attention output (log-sum-exp rescale):
 * M = max_j m_j, out = sum_j e^(m_j - M) o_j / sum_j e^(m_j - M) l_j.
 * [Cohere] "Tasks": ATTN_COMBINE merges the partials into the real output. */
void orc_attend_combine(int d, int parts, const double* m, const double* l, const double* o,
                        double* out) {
  double M = -INFINITY;
  for (int j = 0; j < parts; ++j) M = m[j] > M ? m[j] : M;
  double z = 0.0;
  for (int i = 0; i < d; ++i) out[i] = 0.0;
  for (int j = 0; j < parts; ++j) {
    if (l[j] == 0.0) continue; /* empty slice */
    const double c = exp(m[j] - M);
    z += c * l[j];
    for (int i = 0; i < d; ++i) out[i] += c * o[(size_t)j * d + i];
  }
  for (int i = 0; i < d; ++i) out[i] /= z;
}

/* Top-k of n binary32 logits: ids in descending logit order, equal logits
 * ordered by lower id first.  margin = (k-th) - (k+1-th) logit, +inf when
 * k == n.  [Cohere] "Tasks": ROUTER_TOPK computes the top-k experts of each
 * token. */
int orc_topk(int n, int k, const float* logits, int32_t* ids, float* margin) {
  if (k < 1 || k > n) return -1;
  char* taken = (char*)calloc((size_t)n, 1);
  for (int j = 0; j <= k && j < n; ++j) {
    int best = -1;
    for (int e = 0; e < n; ++e) {
      if (taken[e]) continue;
      if (best < 0 || logits[e] > logits[best]) best = e;
    }
    if (j < k) {
      ids[j] = best;
      taken[best] = 1;
    } else if (margin) {
      *margin = logits[ids[k - 1]] - logits[best];
    }
  }
  if (k == n && margin) *margin = INFINITY;
  free(taken);
  return 0;
}

/* One expert: out = Wd (silu(Wg x) * (Wu x)).  [Cohere] "Tasks": MoE
 * up/gate with the SiLU-and-multiply epilogue, then the down projection. */
void orc_swiglu_expert(const orc_matrix* Wg, const orc_matrix* Wu, const orc_matrix* Wd,
                       const double* x, double* out) {
  const int I = Wg->rows;
  double* g = (double*)malloc(sizeof(double) * (size_t)I);
  double* u = (double*)malloc(sizeof(double) * (size_t)I);
  orc_matvec(Wg, x, g);
  orc_matvec(Wu, x, u);
  for (int i = 0; i < I; ++i) g[i] = orc_silu(g[i]) * u[i];
  orc_matvec(Wd, g, out);
  free(g);
  free(u);
}

/* Routed MoE: out = sum_j w_j expert_{ids_j}(x), j = 0..k-1 in order.
 * [Cohere] "Tasks": MOE_COMBINE sums each token's expert outputs weighted by
 * its router scores.  Matrices are indexed by expert. */
void orc_moe_routed(int k, const int32_t* ids, const double* w, const orc_matrix* Wg,
                    const orc_matrix* Wu, const orc_matrix* Wd, const double* x, double* out) {
  const int H = Wd[0].rows;
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  for (int i = 0; i < H; ++i) out[i] = 0.0;
  for (int j = 0; j < k; ++j) {
    const int e = ids[j];
    orc_swiglu_expert(&Wg[e], &Wu[e], &Wd[e], x, y);
    for (int i = 0; i < H; ++i) out[i] += w[j] * y[i];
  }
  free(y);
}

/* Dense reference for the MoE: every expert evaluated, weighted by a full
 * gate vector (zero outside the routed set gives the routed MoE). */
void orc_moe_dense_gated(int n_experts, const double* gate, const orc_matrix* Wg,
                         const orc_matrix* Wu, const orc_matrix* Wd, const double* x,
                         double* out) {
  const int H = Wd[0].rows;
  double* y = (double*)malloc(sizeof(double) * (size_t)H);
  for (int i = 0; i < H; ++i) out[i] = 0.0;
  for (int e = 0; e < n_experts; ++e) {
    orc_swiglu_expert(&Wg[e], &Wu[e], &Wd[e], x, y);
    for (int i = 0; i < H; ++i) out[i] += gate[e] * y[i];
  }
  free(y);
}

/* Paged KV indexing: logical page = pos / P, offset = pos % P, physical page
 * = block_row[logical page].  [tiny-vllm] "Gathering K/V into a batched
 * buffer and scattering into blocks".  Returns -1 if the page is missing. */
int orc_kv_slot(int64_t pos, int page_size, const int32_t* block_row, int max_pages,
                int32_t* page, int32_t* offset) {
  const int64_t lp = pos / page_size;
  if (pos < 0 || lp >= max_pages || block_row[lp] < 0) return -1;
  *page = block_row[lp];
  *offset = (int32_t)(pos % page_size);
  return 0;
}

/* ------------------------------------------------ the synthetic model */

double orc_e4m3_value(int code) {
  const int e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = e ? ldexp(1.0 + m / 8.0, e - 7) : ldexp(m / 8.0, -6);
  return (code & 0x80) ? -v : v;
}

double orc_e2m1_value(int code) {
  const int e = (code >> 1) & 3, m = code & 1;
  const double v = e ? ldexp(1.0 + m / 2.0, e - 1) : m / 2.0;
  return (code & 8) ? -v : v;
}

void orc_synth_row(const void* ctx, int row, double* out) {
  const orc_synth_src* s = (const orc_synth_src*)ctx;
  const uint64_t key = synth_key(s->seed, synth_stream((uint32_t)s->kind, (uint32_t)s->layer,
                                                       (uint32_t)s->expert));
  if (s->cfg->expert_fp8 && (s->kind == SYNTH_WG || s->kind == SYNTH_WU || s->kind == SYNTH_WD)) {
    /* an FP8 expert row: its E4M3 codes times the row's scale */
    const int skind = s->kind == SYNTH_WG ? SYNTH_SG : s->kind == SYNTH_WU ? SYNTH_SU : SYNTH_SD;
    const uint64_t skey = synth_key(s->seed, synth_stream((uint32_t)skind, (uint32_t)s->layer,
                                                          (uint32_t)s->expert));
    const double scale = (double)synth_row_scale(skey, (uint64_t)row, synth_fp8_base(s->sigma));
    const uint64_t base = (uint64_t)row * (uint64_t)s->cols;
    for (int c = 0; c < s->cols; ++c) out[c] = orc_e4m3_value(synth_fp8(key, base + (uint64_t)c)) * scale;
    return;
  }
  if (s->cfg->expert_fp4 && (s->kind == SYNTH_WG || s->kind == SYNTH_WU || s->kind == SYNTH_WD)) {
    /* an FP4 expert row: element i of the matrix is nibble i % 2 of byte i / 2;
       each 16 elements of the row share a block scale, the row a row scale */
    const int skind = s->kind == SYNTH_WG ? SYNTH_SG : s->kind == SYNTH_WU ? SYNTH_SU : SYNTH_SD;
    const int bkind = s->kind == SYNTH_WG ? SYNTH_BG : s->kind == SYNTH_WU ? SYNTH_BU : SYNTH_BD;
    const uint64_t skey = synth_key(s->seed, synth_stream((uint32_t)skind, (uint32_t)s->layer,
                                                          (uint32_t)s->expert));
    const uint64_t bkey = synth_key(s->seed, synth_stream((uint32_t)bkind, (uint32_t)s->layer,
                                                          (uint32_t)s->expert));
    const double rscale = (double)synth_row_scale(skey, (uint64_t)row, synth_fp4_base(s->sigma));
    const uint64_t base = (uint64_t)row * (uint64_t)s->cols;
    for (int c = 0; c < s->cols; ++c) {
      const uint64_t i = base + (uint64_t)c;
      const int byte = synth_fp4_byte(key, i / 2);
      const int code = (i & 1) ? byte >> 4 : byte & 15;
      const int bcode = synth_fp4_bscale(bkey, (uint64_t)row * (uint64_t)(s->cols / 16) + (uint64_t)(c / 16));
      out[c] = orc_e2m1_value(code) * orc_e4m3_value(bcode) * rscale;
    }
    return;
  }
  const float scale = synth_scale(s->sigma);
  const uint64_t base = (uint64_t)row * (uint64_t)s->cols;
  for (int c = 0; c < s->cols; ++c)
    out[c] = (double)synth_bf16_to_f32(synth_bf16(key, base + (uint64_t)c, scale));
}

orc_matrix orc_synth_matrix(const orc_config* cfg, uint64_t seed, int kind, int layer, int expert,
                            orc_synth_src* st) {
  const int H = cfg->hidden, nq = cfg->n_q, nkv = cfg->n_kv, d = cfg->head_dim;
  int rows = 0, cols = 0;
  switch (kind) {
    case SYNTH_EMB: rows = cfg->vocab; cols = H; break;
    case SYNTH_WQKV: rows = (nq + 2 * nkv) * d; cols = H; break;
    case SYNTH_WO: rows = H; cols = nq * d; break;
    case SYNTH_WR: rows = cfg->n_experts; cols = H; break;
    case SYNTH_WG: case SYNTH_WU: rows = cfg->inter; cols = H; break;
    case SYNTH_WD: rows = H; cols = cfg->inter; break;
    case SYNTH_WLM: rows = cfg->vocab; cols = H; break;
    default: break;
  }
  st->cfg = cfg;
  st->seed = seed;
  st->kind = kind;
  st->layer = layer;
  st->expert = expert;
  st->cols = cols;
  st->sigma = cfg->weight_sigma;
  orc_matrix m = {orc_synth_row, st, rows, cols};
  return m;
}

int64_t orc_synth_dense(const orc_config* cfg, uint64_t seed, int kind, int layer, int expert, double* out) {
  orc_synth_src st;
  const orc_matrix m = orc_synth_matrix(cfg, seed, kind, layer, expert, &st);
  for (int r = 0; r < m.rows; ++r) m.row(m.ctx, r, out + (int64_t)r * m.cols);
  return (int64_t)m.rows * m.cols;
}

/* Pool layout of one layer: [page][kv head][slot][d] (the layout the decode
 * step's KV pool uses). */
void orc_pool_vec(const orc_config* cfg, uint64_t seed, int is_v, int layer, int page, int head,
                  int slot, double* out) {
  const int d = cfg->head_dim, P = cfg->page_size, nkv = cfg->n_kv;
  const uint64_t key = synth_key(seed, synth_stream(is_v ? SYNTH_VPOOL : SYNTH_KPOOL,
                                                    (uint32_t)layer, 0));
  const float scale = synth_scale(cfg->kv_sigma);
  const uint64_t base = (((uint64_t)page * nkv + (uint64_t)head) * P + (uint64_t)slot) * d;
  for (int i = 0; i < d; ++i)
    out[i] = (double)synth_bf16_to_f32(synth_bf16(key, base + (uint64_t)i, scale));
}

static double round_bf16(double v) {
  const float f = (float)v;
  return (double)synth_bf16_to_f32(synth_f32_to_bf16_rne(f));
}

static int config_ok(const orc_config* c) {
  return c->n_layers > 0 && c->hidden > 0 && c->n_q > 0 && c->n_kv > 0 &&
         c->n_q % c->n_kv == 0 && c->head_dim > 0 && c->head_dim % 2 == 0 &&
         c->n_experts > 0 && c->top_k > 0 && c->top_k <= c->n_experts && c->inter > 0 &&
         c->vocab > 0 && c->page_size > 0 && c->window >= 0 && c->full_period > 0 &&
         !(c->expert_fp8 && c->expert_fp4) && (!c->expert_fp4 || (c->hidden % 16 == 0 && c->inter % 16 == 0));
}

/* One decode step for the requested rows.  The layer is the parallel layer
 * of [Cohere] "1. Reduce wave quantization": with x = RMSNorm(h),
 *   h <- h + W_o attn(x) + MoE(x).
 * The step starts from the token's embedding row and ends with the final
 * RMSNorm and the LM head ([Cohere] "Tasks": QKV, attention, O-proj, router,
 * MoE, residual/RMSNorm, LM head).  The new token sits at pos = seq_len - 1;
 * its K and V are written to the pool before attention reads the slice
 * [lo, seq_len) ([tiny-vllm] "The decode loop": the length includes the
 * token; its K/V is written before the attention call).  lo = 0 for a full
 * layer, max(0, seq_len - window) for a sliding one. */
/* The canonical MoE queue of one layer (see oracle.h).  Counting and the
 * prefix sum are written out; the list is filled by walking the routed
 * entries (b, j) in row-major order, each landing at its expert's next free
 * place, which gives rows by b ascending then j ascending within an expert. */
int orc_route_queue(int batch, int k, int n_experts, const int32_t* ids, int32_t* counts, int32_t* offsets,
                    int32_t* rows, int32_t* active) {
  const int n = batch * k;
  for (int e = 0; e < n_experts; ++e) counts[e] = 0;
  for (int i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= n_experts) return -1;
    ++counts[ids[i]];
  }
  offsets[0] = 0;
  for (int e = 0; e < n_experts; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* next = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_experts > 0 ? n_experts : 1));
  for (int e = 0; e < n_experts; ++e) next[e] = offsets[e];
  for (int i = 0; i < n; ++i) rows[next[ids[i]]++] = i;
  free(next);
  int n_active = 0;
  for (int e = 0; e < n_experts; ++e)
    if (counts[e] > 0) {
      active[3 * n_active + 0] = e;
      active[3 * n_active + 1] = offsets[e];
      active[3 * n_active + 2] = counts[e];
      ++n_active;
    }
  return n_active;
}

/* Element offset of (layer, page, head, slot) in a pool [L][pages][n_kv][P][d]. */
static size_t pool_off(const orc_config* cfg, int64_t num_pages, int layer, int page, int head, int slot) {
  return ((((size_t)layer * (size_t)num_pages + (size_t)page) * (size_t)cfg->n_kv + (size_t)head) *
              (size_t)cfg->page_size + (size_t)slot) * (size_t)cfg->head_dim;
}

int orc_decode_step(const orc_config* cfg, const orc_step_in* in, orc_step_out* out) {
  if (!config_ok(cfg) || !in || !out || in->batch <= 0 || in->n_rows < 0) return -1;
  if ((in->k_pool == NULL) != (in->v_pool == NULL)) return -1;
  if (in->k_pool && in->num_pages < 1) return -1;
  const int L = cfg->n_layers, H = cfg->hidden, nq = cfg->n_q, nkv = cfg->n_kv;
  const int d = cfg->head_dim, E = cfg->n_experts, k = cfg->top_k, V = cfg->vocab;
  const int G = nq / nkv, P = cfg->page_size, R = in->n_rows;
  const int QKV = (nq + 2 * nkv) * d;

  for (int r = 0; r < R; ++r) {
    const int b = in->rows[r];
    if (b < 0 || b >= in->batch) return -1;
    const int s = in->seq_lens[b];
    if (s < 1 || (s + P - 1) / P > in->max_pages) return -1;
    if (in->tokens[b] < 0 || in->tokens[b] >= V) return -1;
    if (in->k_pool) /* every page the row reads must be in the explicit pool */
      for (int j = 0; j < (s + P - 1) / P; ++j) {
        const int32_t pg = in->block_tables[(size_t)b * in->max_pages + j];
        if (pg < 0 || pg >= in->num_pages) return -1;
      }
  }

  double* h = (double*)malloc(sizeof(double) * (size_t)H);
  double* x = (double*)malloc(sizeof(double) * (size_t)H);
  double* qkv = (double*)malloc(sizeof(double) * (size_t)QKV);
  double* attn = (double*)malloc(sizeof(double) * (size_t)nq * d);
  double* o = (double*)malloc(sizeof(double) * (size_t)H);
  double* moe = (double*)malloc(sizeof(double) * (size_t)H);
  double* rl = (double*)malloc(sizeof(double) * (size_t)E);
  float* rl32 = (float*)malloc(sizeof(float) * (size_t)E);
  double* wsel = (double*)malloc(sizeof(double) * (size_t)k);
  double* ssel = (double*)malloc(sizeof(double) * (size_t)k);
  int32_t* own = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
  int32_t* use = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
  orc_synth_src* gsrc = (orc_synth_src*)malloc(sizeof(orc_synth_src) * (size_t)E * 3);
  orc_matrix* Wg = (orc_matrix*)malloc(sizeof(orc_matrix) * (size_t)E);
  orc_matrix* Wu = (orc_matrix*)malloc(sizeof(orc_matrix) * (size_t)E);
  orc_matrix* Wd = (orc_matrix*)malloc(sizeof(orc_matrix) * (size_t)E);

  for (int r = 0; r < R; ++r) {
    const int b = in->rows[r];
    const int s = in->seq_lens[b];
    const int64_t pos = (int64_t)s - 1;
    const int32_t* brow = in->block_tables + (size_t)b * in->max_pages;
    orc_synth_src st;

    /* embedding row of the decoded token */
    orc_matrix emb = orc_synth_matrix(cfg, in->seed, SYNTH_EMB, 0, 0, &st);
    emb.row(emb.ctx, in->tokens[b], h);

    for (int l = 0; l < L; ++l) {
      if (out->hidden) memcpy(out->hidden + ((size_t)l * R + r) * H, h, sizeof(double) * H);
      orc_rmsnorm(H, h, in->norm_gamma ? in->norm_gamma + (size_t)l * H : NULL, cfg->eps, x);

      /* attention branch */
      orc_matrix wqkv = orc_synth_matrix(cfg, in->seed, SYNTH_WQKV, l, 0, &st);
      orc_matvec(&wqkv, x, qkv);
      for (int i = 0; i < nq + nkv; ++i) orc_rope(d, qkv + (size_t)i * d, pos, cfg->rope_base);
      if (out->kv_new)
        memcpy(out->kv_new + ((size_t)l * R + r) * 2 * nkv * d, qkv + (size_t)nq * d,
               sizeof(double) * 2 * nkv * d);
      /* the new entry as the BF16 pool holds it */
      for (int i = nq * d; i < QKV; ++i) qkv[i] = round_bf16(qkv[i]);
      if (in->k_pool) { /* stored at position pos before attention reads the pool */
        int32_t page = 0, off = 0;
        orc_kv_slot(pos, P, brow, in->max_pages, &page, &off);
        for (int g = 0; g < nkv; ++g) {
          const size_t o = pool_off(cfg, in->num_pages, l, page, g, off);
          for (int i = 0; i < d; ++i) {
            in->k_pool[o + i] = synth_f32_to_bf16_rne((float)qkv[(size_t)(nq + g) * d + i]);
            in->v_pool[o + i] = synth_f32_to_bf16_rne((float)qkv[(size_t)(nq + nkv + g) * d + i]);
          }
        }
      }

      const int full = cfg->window == 0 || (l + 1) % cfg->full_period == 0;
      const int64_t lo = full ? 0 : (s - cfg->window > 0 ? s - cfg->window : 0);
      const int n = (int)(s - lo);
      double* K = (double*)malloc(sizeof(double) * (size_t)n * d);
      double* Vv = (double*)malloc(sizeof(double) * (size_t)n * d);
      for (int g = 0; g < nkv; ++g) {
#pragma omp parallel for schedule(static)
        for (int t = 0; t < n; ++t) {
          const int64_t p = lo + t;
          if (in->k_pool) {
            int32_t page = 0, off = 0;
            orc_kv_slot(p, P, brow, in->max_pages, &page, &off);
            const size_t o = pool_off(cfg, in->num_pages, l, page, g, off);
            for (int i = 0; i < d; ++i) {
              K[(size_t)t * d + i] = (double)synth_bf16_to_f32(in->k_pool[o + i]);
              Vv[(size_t)t * d + i] = (double)synth_bf16_to_f32(in->v_pool[o + i]);
            }
          } else if (p == pos) {
            memcpy(K + (size_t)t * d, qkv + (size_t)(nq + g) * d, sizeof(double) * d);
            memcpy(Vv + (size_t)t * d, qkv + (size_t)(nq + nkv + g) * d, sizeof(double) * d);
          } else {
            int32_t page = 0, off = 0;
            orc_kv_slot(p, P, brow, in->max_pages, &page, &off);
            orc_pool_vec(cfg, in->seed, 0, l, page, g, off, K + (size_t)t * d);
            orc_pool_vec(cfg, in->seed, 1, l, page, g, off, Vv + (size_t)t * d);
          }
        }
#pragma omp parallel for schedule(static)
        for (int hq = g * G; hq < (g + 1) * G; ++hq)
          orc_attend(d, n, qkv + (size_t)hq * d, K, Vv, 1.0 / sqrt((double)d),
                     attn + (size_t)hq * d);
      }
      free(K);
      free(Vv);
      if (out->attn) memcpy(out->attn + ((size_t)l * R + r) * nq * d, attn, sizeof(double) * nq * d);
      orc_matrix wo = orc_synth_matrix(cfg, in->seed, SYNTH_WO, l, 0, &st);
      orc_matvec(&wo, attn, o);

      /* MoE branch: router, top-k, weights, experts */
      orc_matrix wr = orc_synth_matrix(cfg, in->seed, SYNTH_WR, l, 0, &st);
      orc_matvec(&wr, x, rl);
      for (int e = 0; e < E; ++e) {
        if (in->router_bias) rl[e] += (double)in->router_bias[e];
        rl32[e] = (float)rl[e];
      }
      float margin = 0.0f;
      orc_topk(E, k, rl32, own, &margin);
      const int32_t* f = in->force_ids ? in->force_ids + ((size_t)l * in->batch + b) * k : NULL;
      for (int j = 0; j < k; ++j) use[j] = f ? f[j] : own[j];
      for (int j = 0; j < k; ++j) ssel[j] = rl[use[j]];
      orc_softmax(k, ssel, wsel);
      for (int e = 0; e < E; ++e) {
        Wg[e] = orc_synth_matrix(cfg, in->seed, SYNTH_WG, l, e, &gsrc[3 * e + 0]);
        Wu[e] = orc_synth_matrix(cfg, in->seed, SYNTH_WU, l, e, &gsrc[3 * e + 1]);
        Wd[e] = orc_synth_matrix(cfg, in->seed, SYNTH_WD, l, e, &gsrc[3 * e + 2]);
      }
      orc_moe_routed(k, use, wsel, Wg, Wu, Wd, x, moe);

      for (int i = 0; i < H; ++i) h[i] = h[i] + o[i] + moe[i];

      const size_t lr = (size_t)l * R + r;
      if (out->ids) memcpy(out->ids + lr * k, use, sizeof(int32_t) * k);
      if (out->own_ids) memcpy(out->own_ids + lr * k, own, sizeof(int32_t) * k);
      if (out->weights) memcpy(out->weights + lr * k, wsel, sizeof(double) * k);
      if (out->margin) out->margin[lr] = margin;
      if (out->router_logits) memcpy(out->router_logits + lr * E, rl32, sizeof(float) * E);
    }
    if (out->hidden) memcpy(out->hidden + ((size_t)L * R + r) * H, h, sizeof(double) * H);

    /* final RMSNorm and LM head */
    orc_rmsnorm(H, h, in->final_gamma, cfg->eps, x);
    orc_matrix wlm = orc_synth_matrix(cfg, in->seed, SYNTH_WLM, 0, 0, &st);
    if (out->logits) orc_matvec(&wlm, x, out->logits + (size_t)r * V);
  }

  free(h); free(x); free(qkv); free(attn); free(o); free(moe); free(rl); free(rl32);
  free(wsel); free(ssel); free(own); free(use); free(gsrc); free(Wg); free(Wu); free(Wd);
  return 0;
}
