// mk_service.cpp -- the host decode service ("The inference engine around
// the kernel"): live sequences, their KV pages, one batch per step through a
// step function, greedy tokens streamed back, parking and retiring.  The
// GPU step (mk_decode_step + device argmax) is at the end of the file.
#include <cuda_runtime.h>

#include <algorithm>
#include <deque>
#include <map>
#include <string>
#include <vector>

#include "../../include/mk_service.h"
#include "mk_host.h"

namespace {

struct Seq {
  int64_t id = 0;
  int32_t state = MK_SEQ_RUNNING, finish = MK_FIN_NONE;
  int32_t n_ctx = 0;  // tokens whose K/V are in the pool
  int32_t n_gen = 0, max_new = 0, stop = -1;
  std::deque<int32_t> pending;  // tokens to feed, in order
  std::vector<int32_t> pages;   // logical page j -> pool page
  uint64_t order = 0;           // admission order (batching priority)
};

}  // namespace

struct mk_service {
  mk_service_cfg cfg;
  mk_step_fn step = nullptr;
  void* ctx = nullptr;
  std::map<int64_t, Seq> seqs;
  std::vector<int32_t> free_pages;  // a stack: the next page handed out is back()
  uint64_t next_order = 0;
  // step buffers
  std::vector<int32_t> tok, len, bt, next;
  std::vector<Seq*> rows;
};

using mk::fail;

namespace {

void retire(mk_service* s, Seq& q, int32_t why) {
  for (auto it = q.pages.rbegin(); it != q.pages.rend(); ++it) s->free_pages.push_back(*it);
  q.pages.clear();
  q.pending.clear();
  q.state = MK_SEQ_FINISHED;
  q.finish = why;
}

Seq* find(mk_service* s, int64_t id) {
  auto it = s->seqs.find(id);
  return it == s->seqs.end() ? nullptr : &it->second;
}
const Seq* find(const mk_service* s, int64_t id) {
  auto it = s->seqs.find(id);
  return it == s->seqs.end() ? nullptr : &it->second;
}

}  // namespace

extern "C" {

int mk_service_create(const mk_service_cfg* cfg, mk_step_fn step, void* ctx, mk_service** out) {
  if (!cfg || !step || !out) return fail(MK_ERR_ARG, "null argument");
  *out = nullptr;
  if (cfg->num_pages < 1 || cfg->page_size < 1 || cfg->max_pages < 1 || cfg->max_batch < 1)
    return fail(MK_ERR_ARG, "service sizes must be positive");
  mk_service* s = new mk_service;
  s->cfg = *cfg;
  s->step = step;
  s->ctx = ctx;
  // handed out in increasing order: page 0 first
  for (int32_t p = cfg->num_pages - 1; p >= 0; --p) s->free_pages.push_back(p);
  s->tok.resize(cfg->max_batch);
  s->len.resize(cfg->max_batch);
  s->next.resize(cfg->max_batch);
  s->bt.resize((size_t)cfg->max_batch * cfg->max_pages);
  *out = s;
  return MK_OK;
}

void mk_service_free(mk_service* s) { delete s; }

int mk_service_add(mk_service* s, int64_t id, const int32_t* prompt, int32_t n_prompt, int32_t max_new,
                   int32_t stop_token) {
  if (!s || (!prompt && n_prompt > 0)) return fail(MK_ERR_ARG, "null argument");
  if (n_prompt < 1 || max_new < 1) return fail(MK_ERR_ARG, "a sequence needs a prompt token and max_new >= 1");
  if (s->seqs.count(id)) return fail(MK_ERR_ARG, "sequence id " + std::to_string(id) + " is in use");
  Seq q;
  q.id = id;
  q.max_new = max_new;
  q.stop = stop_token;
  q.pending.assign(prompt, prompt + n_prompt);
  q.order = s->next_order++;
  s->seqs.emplace(id, std::move(q));
  return MK_OK;
}

int mk_service_step(mk_service* s, int64_t* out_ids, int32_t* out_tokens, int32_t cap, int32_t* n_out) {
  if (!s || !n_out) return fail(MK_ERR_ARG, "null argument");
  *n_out = 0;
  const mk_service_cfg& c = s->cfg;
  if (cap > 0 && (!out_ids || !out_tokens)) return fail(MK_ERR_ARG, "null output arrays");
  // running sequences in admission order; a sequence whose next position
  // starts a page needs a free page, else it waits for a later step
  std::vector<Seq*> cand;
  for (auto& kv : s->seqs)
    if (kv.second.state == MK_SEQ_RUNNING) cand.push_back(&kv.second);
  std::sort(cand.begin(), cand.end(), [](const Seq* a, const Seq* b) { return a->order < b->order; });
  s->rows.clear();
  int32_t need_pages = 0;
  for (Seq* q : cand) {
    if ((int32_t)s->rows.size() == c.max_batch) break;
    const bool new_page = q->n_ctx % c.page_size == 0 && (int32_t)q->pages.size() == q->n_ctx / c.page_size;
    if (new_page && need_pages >= (int32_t)s->free_pages.size()) continue;
    need_pages += new_page ? 1 : 0;
    s->rows.push_back(q);
  }
  const int32_t B = (int32_t)s->rows.size();
  if (B == 0) return 0;
  if (cap < B) return fail(MK_ERR_ARG, "output room for " + std::to_string(cap) + " tokens, " +
                                           std::to_string(B) + " rows run");
  // the rows' inputs; pages are taken from the pool only once the step succeeded
  std::fill(s->bt.begin(), s->bt.begin() + (size_t)B * c.max_pages, -1);
  std::vector<int32_t> taken;
  size_t fp = s->free_pages.size();
  for (int32_t r = 0; r < B; ++r) {
    Seq* q = s->rows[r];
    s->tok[r] = q->pending.front();
    s->len[r] = q->n_ctx + 1;
    int32_t* row = &s->bt[(size_t)r * c.max_pages];
    for (size_t j = 0; j < q->pages.size(); ++j) row[j] = q->pages[j];
    if (q->n_ctx % c.page_size == 0 && (int32_t)q->pages.size() == q->n_ctx / c.page_size) {
      const int32_t pg = s->free_pages[--fp];
      row[q->pages.size()] = pg;
      taken.push_back(pg);
    } else {
      taken.push_back(-1);
    }
  }
  mk::set_error("");
  const int rc = s->step(s->ctx, s->tok.data(), s->len.data(), s->bt.data(), B, c.max_pages, s->next.data());
  if (rc != MK_OK) {  // nothing changes: the step can be retried
    if (mk_last_error()[0] == '\0') mk::set_error("step function returned " + std::to_string(rc));
    return rc < 0 ? rc : MK_ERR_ARG;
  }
  s->free_pages.resize(fp);
  int32_t n = 0;
  for (int32_t r = 0; r < B; ++r) {
    Seq* q = s->rows[r];
    if (taken[r] >= 0) q->pages.push_back(taken[r]);
    q->n_ctx += 1;
    q->pending.pop_front();
    if (!q->pending.empty()) continue;  // still feeding: the output is not a sample
    const int32_t t = s->next[r];
    out_ids[n] = q->id;
    out_tokens[n] = t;
    ++n;
    q->n_gen += 1;
    if (t == q->stop) {
      retire(s, *q, MK_FIN_STOP);
    } else if (q->n_gen >= q->max_new) {
      retire(s, *q, MK_FIN_LENGTH);
    } else if (q->n_ctx >= c.max_pages * c.page_size) {
      retire(s, *q, MK_FIN_CONTEXT);  // no position left for the sample
    } else {
      q->pending.push_back(t);  // fed at the next step
    }
  }
  // a sequence still feeding appended tokens can also run out of context
  for (int32_t r = 0; r < B; ++r) {
    Seq* q = s->rows[r];
    if (q->state == MK_SEQ_RUNNING && q->n_ctx >= c.max_pages * c.page_size) retire(s, *q, MK_FIN_CONTEXT);
  }
  *n_out = n;
  return B;
}

int mk_service_run(mk_service* s, int32_t max_steps, mk_token_fn on_token, void* ctx, int32_t* steps_done) {
  if (!s) return fail(MK_ERR_ARG, "null argument");
  if (steps_done) *steps_done = 0;
  std::vector<int64_t> ids(s->cfg.max_batch);
  std::vector<int32_t> toks(s->cfg.max_batch);
  for (int32_t k = 0; k < max_steps; ++k) {
    int32_t n = 0;
    const int rows = mk_service_step(s, ids.data(), toks.data(), s->cfg.max_batch, &n);
    if (rows < 0) return rows;
    if (rows == 0) break;
    if (steps_done) *steps_done = k + 1;
    if (on_token)
      for (int32_t i = 0; i < n; ++i) on_token(ctx, ids[i], toks[i]);
  }
  return MK_OK;
}

int mk_service_park(mk_service* s, int64_t id) {
  Seq* q = s ? find(s, id) : nullptr;
  if (!q) return fail(MK_ERR_ARG, "no sequence " + std::to_string(id));
  if (q->state != MK_SEQ_RUNNING) return fail(MK_ERR_ARG, "sequence " + std::to_string(id) + " is not running");
  q->state = MK_SEQ_PARKED;
  return MK_OK;
}

int mk_service_resume(mk_service* s, int64_t id, const int32_t* tokens, int32_t n) {
  Seq* q = s ? find(s, id) : nullptr;
  if (!q) return fail(MK_ERR_ARG, "no sequence " + std::to_string(id));
  if (q->state != MK_SEQ_PARKED) return fail(MK_ERR_ARG, "sequence " + std::to_string(id) + " is not parked");
  if (n < 0 || (n > 0 && !tokens)) return fail(MK_ERR_ARG, "bad appended tokens");
  q->pending.insert(q->pending.end(), tokens, tokens + n);
  q->state = MK_SEQ_RUNNING;
  return MK_OK;
}

int mk_service_cancel(mk_service* s, int64_t id) {
  Seq* q = s ? find(s, id) : nullptr;
  if (!q) return fail(MK_ERR_ARG, "no sequence " + std::to_string(id));
  if (q->state == MK_SEQ_FINISHED) return fail(MK_ERR_ARG, "sequence " + std::to_string(id) + " has finished");
  retire(s, *q, MK_FIN_CANCEL);
  return MK_OK;
}

int mk_service_forget(mk_service* s, int64_t id) {
  Seq* q = s ? find(s, id) : nullptr;
  if (!q) return fail(MK_ERR_ARG, "no sequence " + std::to_string(id));
  if (q->state != MK_SEQ_FINISHED) return fail(MK_ERR_ARG, "sequence " + std::to_string(id) + " is live");
  s->seqs.erase(id);
  return MK_OK;
}

int mk_service_query(const mk_service* s, int64_t id, mk_seq_info* info) {
  const Seq* q = s ? find(s, id) : nullptr;
  if (!q || !info) return fail(MK_ERR_ARG, "no sequence " + std::to_string(id));
  info->state = q->state;
  info->finish = q->finish;
  info->n_ctx = q->n_ctx;
  info->n_generated = q->n_gen;
  info->n_pending = (int32_t)q->pending.size();
  info->n_pages = (int32_t)q->pages.size();
  return MK_OK;
}

int32_t mk_service_pages(const mk_service* s, int64_t id, int32_t* pages, int32_t cap) {
  const Seq* q = s ? find(s, id) : nullptr;
  if (!q) return fail(MK_ERR_ARG, "no sequence " + std::to_string(id));
  const int32_t n = (int32_t)q->pages.size();
  for (int32_t j = 0; j < n && j < cap; ++j) pages[j] = q->pages[j];
  return n;
}

int32_t mk_service_free_pages(const mk_service* s) { return s ? (int32_t)s->free_pages.size() : 0; }

int32_t mk_service_live(const mk_service* s) {
  int32_t n = 0;
  if (s)
    for (const auto& kv : s->seqs) n += kv.second.state != MK_SEQ_FINISHED ? 1 : 0;
  return n;
}

}  // extern "C"
