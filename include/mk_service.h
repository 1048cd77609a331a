/* mk_service.h -- a host decode service around mk_decode_step.
 *
 * "Cohere: a serving engine for North Mini Code built around a decode
 * megakernel", section "The inference engine around the kernel": a host
 * loop keeps the live requests, updates their page tables, clears the
 * step's scratch, picks a schedule by the batch and the longest live
 * context, launches the step, samples, streams tokens and retires finished
 * requests; a request can be parked (it leaves the batch and keeps its KV
 * pages) and resumed, picking up what was appended to it meanwhile.
 *
 * The service is host code only.  It calls one decode step through a
 * function pointer (mk_step_fn), so the loop runs and is tested without a
 * GPU; mk_gpu_step is the step on the GPU: mk_decode_step on the caller's
 * KV pools and workspace, then a greedy argmax on the device.
 *
 * Reading of the pages: there is no prefill here.  A request's prompt is fed
 * one token per step (each step writes that token's K/V; the output of the
 * last prompt token is the first sampled token); a sampled token is fed at
 * the sequence's next step.  Sampling is greedy (largest logit, lowest id on
 * ties).  The service is single-threaded: calls on one service must not
 * overlap.
 */
#ifndef MK_SERVICE_H
#define MK_SERVICE_H

#include <stddef.h>
#include <stdint.h>

#include "mk.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mk_service mk_service;
typedef struct mk_gpu_step mk_gpu_step;

/* One decode step as the service calls it, on host arrays:
 *  last_tokens  int32 [batch]: the token each row decodes
 *  seq_lens     int32 [batch]: the row's length including that token
 *  block_tables int32 [batch][max_pages]: pages of the row's positions
 *               (entries past the row's last page are -1)
 *  next_tokens  int32 [batch], written: the greedy token after each row
 * Returns MK_OK or a negative MK_ERR_* code (the service step then fails
 * with it and changes no sequence). */
typedef int (*mk_step_fn)(void* ctx, const int32_t* last_tokens, const int32_t* seq_lens,
                          const int32_t* block_tables, int32_t batch, int32_t max_pages,
                          int32_t* next_tokens);

typedef struct mk_service_cfg {
  int32_t num_pages;  /* KV pool pages the service hands out: ids 0 .. num_pages-1 */
  int32_t page_size;  /* tokens per page */
  int32_t max_pages;  /* block-table width; a sequence holds at most max_pages pages
                         (its context is at most max_pages * page_size tokens) */
  int32_t max_batch;  /* rows per step at most */
} mk_service_cfg;

/* sequence states */
#define MK_SEQ_RUNNING 0  /* in the batch whenever there is room and a page */
#define MK_SEQ_PARKED 1   /* out of the batch; keeps its pages */
#define MK_SEQ_FINISHED 2 /* retired: its pages are back in the pool */

/* why a sequence finished */
#define MK_FIN_NONE 0
#define MK_FIN_LENGTH 1   /* max_new tokens sampled */
#define MK_FIN_STOP 2     /* sampled the stop token (it is emitted) */
#define MK_FIN_CONTEXT 3  /* the context reached max_pages * page_size */
#define MK_FIN_CANCEL 4   /* mk_service_cancel */

typedef struct mk_seq_info {
  int32_t state;        /* MK_SEQ_* */
  int32_t finish;       /* MK_FIN_* */
  int32_t n_ctx;        /* tokens whose K/V are in the pool */
  int32_t n_generated;  /* tokens sampled and emitted */
  int32_t n_pending;    /* tokens waiting to be fed (prompt, the last sample, appended) */
  int32_t n_pages;      /* pages held */
} mk_seq_info;

/* Creates a service; `step` and `ctx` are kept and called by
 * mk_service_step.  MK_ERR_ARG for non-positive sizes or a null step. */
int mk_service_create(const mk_service_cfg* cfg, mk_step_fn step, void* ctx, mk_service** out);
void mk_service_free(mk_service* s);

/* Admits sequence `id` (unique among the service's sequences, finished ones
 * included until mk_service_forget) with its prompt (n_prompt >= 1 tokens,
 * copied).  It is decoded until max_new (>= 1) tokens are sampled or it
 * samples stop_token (< 0: none).  MK_ERR_ARG for a duplicate id or a bad
 * count. */
int mk_service_add(mk_service* s, int64_t id, const int32_t* prompt, int32_t n_prompt, int32_t max_new,
                   int32_t stop_token);

/* One step: takes up to max_batch running sequences in admission order
 * (a sequence that needs a new page when none is free waits for a later
 * step), calls the step function once, advances every row, and retires the
 * sequences that finished (their pages return to the pool).  The sampled
 * tokens are written as (id, token) pairs to out_ids / out_tokens (room for
 * `cap` pairs; at most max_batch are produced) and their count to *n_out.
 * Returns the number of rows decoded (0: no running sequence could run) or
 * a negative error: the step function's, or MK_ERR_ARG for cap too small. */
int mk_service_step(mk_service* s, int64_t* out_ids, int32_t* out_tokens, int32_t cap, int32_t* n_out);

/* The loop itself: steps until no running sequence can run or max_steps
 * steps were taken, handing each sampled token to on_token (may be NULL) as
 * it is produced.  *steps_done (may be NULL) gets the steps taken.  Returns
 * MK_OK or the first failing step's error (the sequences are as before that
 * step). */
typedef void (*mk_token_fn)(void* ctx, int64_t id, int32_t token);
int mk_service_run(mk_service* s, int32_t max_steps, mk_token_fn on_token, void* ctx, int32_t* steps_done);

/* Parks a running sequence (it keeps its pages and pending tokens). */
int mk_service_park(mk_service* s, int64_t id);
/* Resumes a parked sequence, first appending n >= 0 tokens (copied) to its
 * pending tokens: they are fed after what was pending (the last sample),
 * and sampling resumes after the last of them. */
int mk_service_resume(mk_service* s, int64_t id, const int32_t* tokens, int32_t n);
/* Retires a running or parked sequence (MK_FIN_CANCEL); its pages return. */
int mk_service_cancel(mk_service* s, int64_t id);
/* Drops a finished sequence's record (its id may then be reused). */
int mk_service_forget(mk_service* s, int64_t id);

int mk_service_query(const mk_service* s, int64_t id, mk_seq_info* info);
/* The sequence's pages in logical order (at most cap); returns their count. */
int32_t mk_service_pages(const mk_service* s, int64_t id, int32_t* pages, int32_t cap);
int32_t mk_service_free_pages(const mk_service* s);
int32_t mk_service_live(const mk_service* s); /* running + parked */

/* ---- the step on the GPU ---- */

/* Device bytes mk_gpu_step needs for its inputs and outputs at this batch
 * and block-table width (tokens, lengths and block tables as one block; the
 * next tokens and a copy of the step's error record; fp32 logits),
 * 256-byte aligned parts.  The GPU step also holds pinned host copies of
 * the input and output blocks (one copy each way per step). */
size_t mk_gpu_step_dev_bytes(const mk_model* m, int32_t max_batch, int32_t max_pages);

/* A GPU step on the caller's memory: the KV pools ([n_layers][num_pages]
 * [n_kv][page_size][head_dim] bf16), a workspace of at least the largest
 * mk_workspace_bytes of the schedules, and dev_buf of
 * mk_gpu_step_dev_bytes(m, largest max_batch, max_pages).  `scheds` are
 * uploaded schedules (mk_sched_upload); each step uses the first one whose
 * max_batch and max_ctx cover the batch and its longest row ("The inference
 * engine around the kernel": a schedule per context bucket).  The handles
 * are kept, not owned.  Use mk_gpu_step_run with the handle as ctx. */
int mk_gpu_step_create(mk_model* m, mk_sched* const* scheds, int32_t n_scheds, void* k_pool, void* v_pool,
                       int64_t num_pages, int32_t max_pages, void* workspace, size_t workspace_bytes,
                       void* dev_buf, size_t dev_bytes, void* stream, mk_gpu_step** out);
void mk_gpu_step_free(mk_gpu_step* g);

/* mk_step_fn for ctx = an mk_gpu_step: copies the inputs to the device,
 * runs mk_decode_step and the argmax on the stream, copies the tokens back
 * and waits; device-side failures come back as mk_check_step's code.
 * MK_ERR_ARG when no schedule covers the batch.  The first step of each
 * (schedule, batch) is captured as a CUDA graph that later steps replay with
 * one launch; on a stream that cannot be captured (the legacy default
 * stream) the steps are issued one by one. */
int mk_gpu_step_run(void* ctx, const int32_t* last_tokens, const int32_t* seq_lens,
                    const int32_t* block_tables, int32_t batch, int32_t max_pages, int32_t* next_tokens);

/* Greedy token of each row of fp32 logits [rows][vocab] (largest value,
 * lowest index on ties; NaN never wins) into next [rows], on the stream. */
int mk_argmax_rows(const float* logits, int32_t rows, int32_t vocab, int32_t* next, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MK_SERVICE_H */
