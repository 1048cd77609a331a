/*
 * oracle.h -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * A plain, slow, fp64 CPU statement of one decode step of a parallel
 * attention / MoE transformer, written from the text of "Cohere: a decode
 * megakernel for North Mini Code" (the parallel layer of section "1. Reduce
 * wave quantization"; the operations listed under "Tasks") and, for the
 * formulas those pages leave out (RoPE angles, the position of the new KV
 * entry, paged indexing, online softmax), from "tiny-vllm 5: the decode path"
 * (sections "RoPE", "Gathering K/V into a batched buffer", "Attention is
 * finished off by pagedAttentionKernel").
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  It shares no code with the GPU path; the one thing both
 * compile is the input generator synth/synth.h.
 *
 * Precision: inputs (weights, KV) are BF16 and are upcast exactly; every sum
 * is accumulated in double in index order.  Two roundings are part of the
 * definition, not of the arithmetic: the new token's K and V are stored in the
 * BF16 pool before attention reads them, and the router logits are rounded to
 * binary32 before the top-k decision (the precision the GPU decides in).
 */
#ifndef MK_ORACLE_H
#define MK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int n_layers, hidden, n_q, n_kv, head_dim, n_experts, top_k, inter, vocab;
  int page_size;
  int window;      /* 0: no sliding window */
  int full_period; /* layer l attends to the whole context iff window == 0 or (l+1) % full_period == 0 */
  double rope_base, eps, weight_sigma, kv_sigma;
  int expert_fp8;  /* 1: expert matrices are E4M3 codes times one scale per output row */
  int expert_fp4;  /* 1: expert matrices are E2M1 codes times an E4M3 scale per 16 inputs
                      times one scale per output row */
} orc_config;

/* FP4 E2M1 code (4 bits) -> value: (-1)^s 2^(e-1) (1 + m/2) for exponent field
 * e > 0, (-1)^s m/2 for e = 0 (1 sign, 2 exponent, 1 mantissa bit). */
double orc_e2m1_value(int code);

/* OCP FP8 E4M3 code -> value: (-1)^s 2^(e-7) (1 + m/8) for exponent field
 * e > 0, (-1)^s 2^-6 (m/8) for e = 0 (1 sign, 4 exponent, 3 mantissa bits;
 * no infinities; codes 0x7f and 0xff are NaN). */
double orc_e4m3_value(int code);

/* A matrix given row by row: row(ctx, r, out) writes the `cols` doubles of row r. */
typedef void (*orc_row_fn)(const void* ctx, int row, double* out);

typedef struct {
  orc_row_fn row;
  const void* ctx;
  int rows, cols;
} orc_matrix;

/* A dense row-major double matrix as a row source (ctx = orc_dense*). */
typedef struct {
  const double* data;
  int cols;
} orc_dense;
void orc_dense_row(const void* ctx, int row, double* out);

/* ---- the operations of one layer, each on explicit operands ---- */
void orc_rmsnorm(int n, const double* x, const double* gamma, double eps, double* out);
void orc_rope(int d, double* v, int64_t pos, double base);
void orc_softmax(int n, const double* s, double* p);
double orc_silu(double x);
void orc_matvec(const orc_matrix* W, const double* x, double* y);
void orc_attend(int d, int n, const double* q, const double* K, const double* V, double scale,
                double* out);
void orc_attend_partial(int d, int n, const double* q, const double* K, const double* V,
                        double scale, double* m, double* l, double* o);
void orc_attend_combine(int d, int parts, const double* m, const double* l, const double* o,
                        double* out);
int orc_topk(int n, int k, const float* logits, int32_t* ids, float* margin);
void orc_swiglu_expert(const orc_matrix* Wg, const orc_matrix* Wu, const orc_matrix* Wd,
                       const double* x, double* out);
void orc_moe_routed(int k, const int32_t* ids, const double* w, const orc_matrix* Wg,
                    const orc_matrix* Wu, const orc_matrix* Wd, const double* x, double* out);
void orc_moe_dense_gated(int n_experts, const double* gate, const orc_matrix* Wg,
                         const orc_matrix* Wu, const orc_matrix* Wd, const double* x,
                         double* out);
int orc_kv_slot(int64_t pos, int page_size, const int32_t* block_row, int max_pages,
                int32_t* page, int32_t* offset);

/* ---- the synthetic model: weights and the initial KV pool regenerated on demand ---- */
typedef struct {
  const orc_config* cfg;
  uint64_t seed;
  int kind, layer, expert, cols;
  double sigma;
} orc_synth_src;
void orc_synth_row(const void* ctx, int row, double* out);
orc_matrix orc_synth_matrix(const orc_config* cfg, uint64_t seed, int kind, int layer, int expert,
                            orc_synth_src* storage);
/* The whole matrix of a weight kind as the oracle reads it, row-major into out
 * (rows * cols doubles); returns rows * cols. */
int64_t orc_synth_dense(const orc_config* cfg, uint64_t seed, int kind, int layer, int expert, double* out);
/* K (is_v = 0) or V (is_v = 1) of one pool slot, as the generator filled it. */
void orc_pool_vec(const orc_config* cfg, uint64_t seed, int is_v, int layer, int page, int head,
                  int slot, double* out);

typedef struct {
  uint64_t seed;
  int batch;
  const int32_t* tokens;       /* [B] token decoded this step */
  const int32_t* seq_lens;     /* [B] sequence length including that token */
  const int32_t* block_tables; /* [B][max_pages] physical page of each logical page */
  int max_pages;
  const float* router_bias;    /* [E] added to the router logits, or NULL */
  const int32_t* force_ids;    /* [L][B][k] routing to follow, or NULL (see orc_decode_step) */
  int n_rows;
  const int32_t* rows;         /* the batch rows b to evaluate */
  const double* norm_gamma;    /* [L][H] gain of each layer's input RMSNorm, or NULL (all ones) */
  const double* final_gamma;   /* [H] gain of the final RMSNorm, or NULL (all ones) */
  /* Optional explicit KV pools, BF16 bit patterns [L][num_pages][n_kv][P][d]
   * (K and V).  NULL: the generator's pool, never written.  Given: attention
   * reads every key and value from them through the block table, and the
   * step first stores the new token's K and V (rounded to BF16) in the slot
   * of position seq_len - 1, so that a later call sees what this one wrote. */
  uint16_t* k_pool;
  uint16_t* v_pool;
  int64_t num_pages;
} orc_step_in;

typedef struct {
  double* logits;       /* [n_rows][V] */
  int32_t* ids;         /* [L][n_rows][k] experts used (descending logit) */
  double* weights;      /* [L][n_rows][k] their router weights */
  int32_t* own_ids;     /* [L][n_rows][k] the oracle's own top-k */
  float* margin;        /* [L][n_rows] k-th minus (k+1)-th binary32 router logit */
  float* router_logits; /* [L][n_rows][E] binary32 */
  double* hidden;       /* optional [L+1][n_rows][H]: residual entering each layer, then the last */
  double* kv_new;       /* optional [L][n_rows][2][n_kv][d]: new K (after RoPE) and V, before BF16 */
  double* attn;         /* optional [L][n_rows][n_q d]: attention output */
} orc_step_out;

/* The MoE work queue of one layer, as ROUTE_FINALIZE builds it ("Cohere: a
 * decode megakernel for North Mini Code", section "Tasks": the routing
 * becomes per-expert row counts and offsets and the expert-ordered list of
 * routed rows that the MoE GEMM tiles drain).  ids [batch][k] are the experts
 * of each row.  Canonical order: experts ascending; within an expert, routed
 * entries by row b ascending, then choice j ascending.
 *   counts  [n_experts]      rows routed to each expert
 *   offsets [n_experts + 1]  exclusive prefix sum of counts (offsets[E] = batch * k)
 *   rows    [batch * k]      entry i of the expert-ordered list is b * k + j
 *   active  [n_experts][3]   the experts with rows, ascending: {expert, offset, count}
 * Returns the number of active experts, or -1 on an expert id out of range. */
int orc_route_queue(int batch, int k, int n_experts, const int32_t* ids, int32_t* counts, int32_t* offsets,
                    int32_t* rows, int32_t* active);

/* Returns 0, or -1 on an invalid argument.  With force_ids, layer l of row
 * b uses the forced experts instead of its own top-k; the caller is the one
 * who checks that the forced set differs from the oracle's only at a
 * near-tie (margin). */
int orc_decode_step(const orc_config* cfg, const orc_step_in* in, orc_step_out* out);

#ifdef __cplusplus
}
#endif
#endif
