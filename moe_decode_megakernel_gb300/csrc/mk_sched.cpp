// mk_sched.cpp -- the host task scheduler: builds the per-SM task lists of
// one decode step, validates them, and simulates them on the host.
//
// "Cohere: a decode megakernel for North Mini Code", section "Task
// scheduler": the host builds named waves per layer, puts them in a chosen
// order, flattens them into one list and assigns task k to SM k mod #SMs;
// full attention and the MoE, whose sizes depend on live sequence lengths and
// routing, are drained from shared queues by a fixed number of claimer tasks.
// Section "How do you write a megakernel?": a wrong arrive count drifts warps
// onto other tasks and deadlocks much later, so barrier accounting gets
// explicit invariants -- the validator and the simulator below.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <deque>
#include <map>
#include <random>
#include <sstream>

#include "mk_host.h"

namespace mk {

bool is_full_layer(const mk_config& c, int l) {
  return c.window == 0 || (l + 1) % c.full_period == 0;
}

int attn_slices(const mk_sched* s, int seq_len) {
  return (seq_len + s->split_len - 1) / s->split_len;
}

size_t WsLayout::off(const char* name) const {
  for (auto& r : regions)
    if (r.first == name) return r.second;
  return (size_t)-1;
}

size_t WsLayout::add(const char* name, size_t bytes) {
  total = (total + 255) & ~(size_t)255;
  regions.emplace_back(name, total);
  size_t o = total;
  total += bytes;
  return o;
}

namespace {

Desc blank(int op, int layer) {
  Desc d;
  d.fill(0);
  d[F_OP] = op;
  d[F_LAYER] = layer;
  d[F_WAIT0] = d[F_WAIT1] = -1;
  d[F_SIG0] = d[F_SIG1] = -1;
  return d;
}

struct Builder {
  mk_sched* s;
  int MB, L, E, NKV, K;
  int nbars = 0;

  int bar(BarKind k, int n = 1) {
    int b = nbars;
    nbars += n;
    for (int i = 0; i < n; ++i) s->bar_kind.push_back(k);
    return b;
  }

  void alloc_layer_bars() {
    s->lb.assign(L + 1, LayerBars());
    for (int l = 0; l <= L; ++l) {
      LayerBars& b = s->lb[l];
      b.norm = bar(BK_STATIC);
      if (l == L) break;
      b.qkv = bar(BK_STATIC, NKV);
      b.router = bar(BK_STATIC);
      b.topk = bar(BK_STATIC);
      b.fin = bar(BK_STATIC);
      if (s->opts.explicit_gather) b.gather = bar(BK_STATIC);
      b.cnt = bar(BK_ATTN_COUNT, MB * NKV);
      b.acomb = bar(BK_STATIC, NKV);
      b.up = bar(BK_UP_EXPERT, E);
      b.upd = bar(BK_STATIC);
      b.dnd = bar(BK_STATIC);
      if (!s->opts.fuse_moe_combine) b.mcomb = bar(BK_STATIC);
      b.o = bar(BK_STATIC);
      b.attn_done = bar(BK_STATIC);
      b.claim_attn = bar(BK_CLAIM);
      b.claim_up = bar(BK_CLAIM);
      b.claim_dn = bar(BK_CLAIM);
      b.rarrive = bar(BK_CLAIM);
    }
    s->lm_bar = bar(BK_STATIC);
  }

  static void wait(Desc& d, int slot, int b, int tgt) {
    d[slot == 0 ? F_WAIT0 : F_WAIT1] = b;
    d[slot == 0 ? F_TGT0 : F_TGT1] = tgt;
  }

  // -------- waves of one layer
  std::vector<Desc> norm_wave(int l, int rows_per_task) {
    std::vector<Desc> w;
    LayerBars& b = s->lb[l];
    for (int b0 = 0; b0 < MB; b0 += rows_per_task) {
      Desc d = blank(OP_RESID_NORM, l);
      d[F_A0] = b0;
      d[F_A0 + 1] = std::min(MB, b0 + rows_per_task);
      d[F_A0 + 2] = (l == L);
      d[F_A0 + 3] = s->opts.fuse_moe_combine;
      if (l > 0) {
        LayerBars& p = s->lb[l - 1];
        wait(d, 0, p.o, p.n_o);
        if (s->opts.fuse_moe_combine) wait(d, 1, p.dnd, p.n_dn_claim);
        else wait(d, 1, p.mcomb, p.n_mcomb);
      }
      d[F_SIG0] = b.norm;
      w.push_back(d);
    }
    b.n_norm = (int)w.size();
    return w;
  }

  std::vector<Desc> dense_wave(int op, int l, int rows, int tile, int sig) {
    std::vector<Desc> w;
    for (int r0 = 0; r0 < rows; r0 += tile) {
      Desc d = blank(op, l);
      d[F_A0] = r0;
      d[F_A0 + 1] = std::min(tile, rows - r0);
      d[F_SIG0] = sig;
      w.push_back(d);
    }
    return w;
  }
};

int auto_split_pages(const mk_sched* s) {
  if (s->opts.attn_split_pages > 0) return s->opts.attn_split_pages;
  const int P = s->cfg.page_size;
  // about one KV slice per SM for a full-attention layer at the largest batch and context
  // (full shape, batch 1, 8K: 4 pages; 2 pages, twice the slices to merge, measured 3% slower),
  // and no slice above 1 MB of K/V: one SM streams such a slice for 15 us or more, so larger
  // ones leave the SMs unbalanced (ragged batch 32 at up to 32K: 10.9 ms with 64-page slices,
  // 10.0 ms with 32-page ones; ragged batch 64 at up to 64K: 24.1 and 24.4 ms)
  const double tok = (double)s->max_batch * s->cfg.n_kv * s->max_ctx / (double)s->num_sms;
  const int most = std::max(1, std::min(64, (int)((1 << 20) / ((int64_t)P * s->cfg.head_dim * 2 * 2))));
  int pages = (int)((tok + P - 1) / P);
  return std::max(1, std::min(pages, most));
}

// Static MoE claims by readiness: the claimer of rank r takes units r, r + n,
// ..., so the lowest ranks get the extra units.  The ranks go to the SMs that
// reach their claimer earliest, estimated by walking the layer's tasks in
// list order (task k runs on SM k mod n) with each task starting no earlier
// than its inputs are typically ready and taking its typical busy time (the
// full shape's measured values, 0.1 us, from the layer's start); the up/gate
// ranks first, then the down ranks with the up/gate units counted in.
void balance_moe_ranks(mk_sched* s, std::vector<Desc>& all, size_t begin, int MB, bool full) {
  const int n = s->num_sms;
  const ShapeDims& D = s->dims;
  const int U = s->plan.up_tiles, DN = s->plan.dn_tiles;
  const int n_act = std::min(D.E, MB * D.K);  // fewest active experts: one row's K
  const int64_t up_units = (int64_t)n_act * U, dn_units = (int64_t)n_act * DN;
  const int64_t attn_entries = (int64_t)MB * D.NKV * ((s->max_ctx + s->split_len - 1) / s->split_len);
  std::vector<int> up_rank(n, -1), dn_rank(n, -1);
  std::vector<int64_t> at_up(n, 0), at_dn(n, 0);
  std::vector<size_t> up_at(n, SIZE_MAX), dn_at(n, SIZE_MAX);
  auto units_of = [](int r, int64_t units, int nc) -> int64_t { return r < units ? (units - r + nc - 1) / nc : 0; };
  auto walk = [&]() {
    std::vector<int64_t> t(n, 0);
    for (size_t k = begin; k < all.size(); ++k) {
      const Desc& d = all[k];
      const int sm = (int)(k % (size_t)n);
      int64_t earliest = 0, dur = 0;
      switch (d[F_OP]) {
        case OP_RESID_NORM: dur = 24; break;
        case OP_ROUTER_GEMM: dur = 60; break;
        case OP_QKV_PROJ: dur = 55; break;
        case OP_ATTN_DECODE: earliest = 75; dur = 56; break;
        case OP_ATTN_DRAIN: {
          const int64_t ci = d[F_A0 + 4], nc = std::max(1, d[F_A0 + 5]);
          earliest = 75;
          dur = 64 * (ci >= 0 ? units_of((int)ci, attn_entries, (int)nc) : (attn_entries + nc - 1) / nc);
          break;
        }
        case OP_ATTN_COMBINE: earliest = full ? 155 : 145; dur = 50; break;
        case OP_O_PROJ: earliest = 215; dur = 25; break;
        case OP_MOE_UPGATE_ACT_DRAIN:
          up_at[sm] = k;
          at_up[sm] = std::max(t[sm], (int64_t)90);
          t[sm] = at_up[sm] + (up_rank[sm] >= 0 ? 60 * units_of(up_rank[sm], up_units, n) : 0);
          continue;
        case OP_MOE_DOWN_DRAIN:
          dn_at[sm] = k;
          at_dn[sm] = std::max(t[sm], (int64_t)190);
          t[sm] = at_dn[sm] + (dn_rank[sm] >= 0 ? 23 * units_of(dn_rank[sm], dn_units, n) : 0);
          continue;
        default: break;
      }
      t[sm] = std::max(t[sm], earliest) + dur;
    }
  };
  auto rank = [&](std::vector<size_t>& at, std::vector<int64_t>& when, std::vector<int>& out) {
    std::vector<int> order;
    for (int sm = 0; sm < n; ++sm)
      if (at[sm] != SIZE_MAX) order.push_back(sm);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return when[a] < when[b]; });
    for (int r = 0; r < (int)order.size(); ++r) {
      Desc& d = all[at[order[r]]];
      d[F_A0 + 4] = r;
      d[F_A0 + 7] = 2;  // static by rank, no shift of the down units
      out[order[r]] = r;
    }
  };
  walk();
  rank(up_at, at_up, up_rank);
  walk();
  rank(dn_at, at_dn, dn_rank);
}

// Greedy placement ("Task scheduler": the cost-model scheduler the pages
// tried before round robin): each layer's tasks, in list order, go one by one
// to the SM where they are estimated to finish first, every SM starting the
// layer at time 0.  A task's estimate is its typical input-ready time and
// busy time at the full shape (0.1 us; a claimer's busy time is its static
// units times one unit's), scaled by its weight bytes for GEMV tiles of other
// sizes.  Each SM's list stays in list order, so every wait still points to
// an earlier task.
std::vector<int> place_greedy(const mk_sched* s, const std::vector<Desc>& all,
                              const std::vector<size_t>& layer_begin, int MB) {
  const int n = s->num_sms;
  const ShapeDims& D = s->dims;
  const int U = s->plan.up_tiles, DN = s->plan.dn_tiles;
  const int n_act = std::min(D.E, MB * D.K);
  const int64_t up_units = (int64_t)n_act * U, dn_units = (int64_t)n_act * DN;
  auto units_of = [](int64_t r, int64_t units, int64_t nc) -> int64_t {
    return r >= 0 && r < units ? (units - r + nc - 1) / nc : 0;
  };
  std::vector<int> sm_of(all.size(), 0);
  std::vector<int64_t> t(n, 0);
  for (size_t li = 0; li < layer_begin.size(); ++li) {
    const size_t b = layer_begin[li], e = li + 1 < layer_begin.size() ? layer_begin[li + 1] : all.size();
    std::fill(t.begin(), t.end(), 0);
    const bool full = is_full_layer(s->cfg, (int)li);
    const int64_t entries = (int64_t)MB * D.NKV * ((s->max_ctx + s->split_len - 1) / s->split_len);
    for (size_t k = b; k < e; ++k) {
      const Desc& d = all[k];
      int64_t earliest = 0, dur = 10;
      const int64_t nc = std::max(1, d[F_A0 + 5]);
      switch (d[F_OP]) {
        case OP_RESID_NORM: dur = 24; break;
        case OP_ROUTER_GEMM: dur = 60; break;
        case OP_QKV_PROJ: dur = 55; break;
        case OP_ATTN_DECODE: earliest = 75; dur = 56; break;
        case OP_ATTN_DRAIN: earliest = 75; dur = 64 * units_of(d[F_A0 + 4], entries, nc); break;
        case OP_ATTN_COMBINE: earliest = full ? 155 : 145; dur = 50; break;
        case OP_O_PROJ: earliest = 215; dur = 25; break;
        case OP_MOE_UPGATE_ACT_DRAIN: earliest = 90; dur = 90 * units_of(d[F_A0 + 4], up_units, nc); break;
        case OP_MOE_DOWN_DRAIN: earliest = 190; dur = 24 * units_of(d[F_A0 + 4], dn_units, nc); break;
        case OP_FFN_UPGATE_ACT: earliest = 30; dur = 60; break;
        case OP_FFN_DOWN: earliest = 90; dur = 30; break;
        case OP_LM_HEAD: dur = 40; break;
        default: break;
      }
      // ties (zero-cost claimers, an idle start) go round robin from task k's own SM
      int best = (int)(k % (size_t)n);
      int64_t best_end = INT64_MAX;
      for (int i = 0; i < n; ++i) {
        const int sm = (int)((k + (size_t)i) % (size_t)n);
        const int64_t end = std::max(t[sm], earliest) + dur;
        if (end < best_end) {
          best_end = end;
          best = sm;
        }
      }
      sm_of[k] = best;
      t[best] = best_end;
    }
  }
  return sm_of;
}

// Split placement: the two branches of the parallel layer ("1. Reduce wave
// quantization": attention and the MoE read the same normalised input and
// rejoin at the residual) on disjoint SMs.  Each branch's tasks keep their
// list order and go round robin over the branch's SMs, so a wait in one
// branch never holds a task of the other; the LM head (after the last layer)
// goes over every SM.
std::vector<int> place_split(const mk_sched* s, const std::vector<Desc>& all, const std::vector<size_t>& layer_begin,
                             int n_attn) {
  const int n = s->num_sms, n_moe = n - n_attn;
  std::vector<int> sm_of(all.size(), 0);
  const size_t lm_begin = layer_begin.back();  // the final RMSNorm, then the LM head
  int64_t ca = 0, cm = 0, cl = 0;
  for (size_t k = 0; k < all.size(); ++k) {
    const int op = all[k][F_OP];
    if (k >= lm_begin && op == OP_LM_HEAD) {
      sm_of[k] = (int)(cl++ % n);
      continue;
    }
    const bool attn = op == OP_QKV_PROJ || op == OP_ATTN_DECODE || op == OP_ATTN_DRAIN || op == OP_ATTN_COMBINE ||
                      op == OP_O_PROJ;
    sm_of[k] = attn ? (int)(ca++ % n_attn) : n_attn + (int)(cm++ % n_moe);
  }
  return sm_of;
}

// Dependency-affinity placement ("Task scheduler": placing a task on the SM
// that produced its input, which the pages measured 1-2% slower than round
// robin): each layer's tasks in list order go to an SM among those that ran
// a task signalling one of the barriers the task waits on, the least loaded
// of them, provided it holds fewer than `cap` of the layer's tasks (the
// layer's tasks per SM, rounded up); otherwise to the least loaded SM, round
// robin among equals.  The fused routing barrier counts the router tasks as
// its signallers.
std::vector<int> place_affinity(const mk_sched* s, const std::vector<Desc>& all,
                                const std::vector<size_t>& layer_begin) {
  const int n = s->num_sms;
  const int NB = (int)s->bar_kind.size();
  std::vector<int> sm_of(all.size(), 0);
  std::vector<std::vector<int>> sig_sms(NB);  // barrier -> SMs of its signallers so far
  std::vector<int> load(n, 0);
  int rr = 0;
  for (size_t li = 0; li < layer_begin.size(); ++li) {
    const size_t b = layer_begin[li], e = li + 1 < layer_begin.size() ? layer_begin[li + 1] : all.size();
    std::fill(load.begin(), load.end(), 0);
    const int cap = (int)((e - b + n - 1) / n);
    for (size_t k = b; k < e; ++k) {
      const Desc& d = all[k];
      int best = -1;
      for (int f : {F_WAIT0, F_WAIT1}) {
        const int bar = d[f];
        if (bar < 0 || bar >= NB) continue;
        for (int sm : sig_sms[bar])
          if (load[sm] < cap && (best < 0 || load[sm] < load[best])) best = sm;
      }
      if (best < 0) {  // no producer SM with room: the least loaded SM, round robin among equals
        for (int i = 0; i < n; ++i) {
          const int sm = (rr + i) % n;
          if (best < 0 || load[sm] < load[best]) best = sm;
        }
        rr = (best + 1) % n;
      }
      sm_of[k] = best;
      ++load[best];
      for (int f : {F_SIG0, F_SIG1})
        if (d[f] >= 0 && d[f] < NB) sig_sms[d[f]].push_back(best);
      if (d[F_OP] == OP_ROUTER_GEMM && d[F_A0 + 5] && d[F_A0 + 4] >= 0 && d[F_A0 + 4] < NB)
        sig_sms[d[F_A0 + 4]].push_back(best);
    }
  }
  return sm_of;
}

// Slices where there are no up/gate tiles: round robin, except that the
// static attention slices of each layer go first to the SMs whose up/gate
// claimer gets no unit (at batch 1 the routed experts' up/gate tiles are
// fewer than the claimers), at most `cap` each, so that no slice delays an
// SM's up/gate tile.  Applies where the claims are static.
std::vector<int> place_slices_free(const mk_sched* s, const std::vector<Desc>& all,
                                   const std::vector<size_t>& layer_begin, int MB, int cap) {
  const int n = s->num_sms;
  std::vector<int> sm_of(all.size());
  for (size_t k = 0; k < all.size(); ++k) sm_of[k] = (int)(k % (size_t)n);
  const int64_t up_units = (int64_t)std::min(s->dims.E, MB * s->dims.K) * s->plan.up_tiles;
  for (size_t li = 0; li + 1 < layer_begin.size(); ++li) {
    const size_t b = layer_begin[li], e = layer_begin[li + 1];
    std::vector<int> free_sms;
    for (size_t k = b; k < e; ++k) {
      const Desc& d = all[k];
      if (d[F_OP] == OP_MOE_UPGATE_ACT_DRAIN && d[F_A0 + 7] == 1 && d[F_A0 + 4] >= up_units)
        free_sms.push_back(sm_of[k]);
    }
    if (free_sms.empty()) continue;
    size_t given = 0;
    for (size_t k = b; k < e && given < free_sms.size() * (size_t)cap; ++k)
      if (all[k][F_OP] == OP_ATTN_DECODE) sm_of[k] = free_sms[given++ % free_sms.size()];
  }
  return sm_of;
}

}  // namespace

// SMs of the attention branch under the split placement (all SMs otherwise):
// opts.attn_sms, or the branch's share of a layer's bytes at the schedule's
// largest batch and context (QKV, O-proj and the KV it reads against the
// router and the experts the batch can route to).
int attn_group_sms(const mk_sched* s) {
  if (s->opts.placement != 2) return s->num_sms;
  const ShapeDims& D = s->dims;
  const mk_config& c = s->cfg;
  const int n = s->num_sms;
  int a = s->opts.attn_sms;
  if (a <= 0) {
    const double eb = c.expert_fp4 ? 0.5 + 1.0 / 16 : c.expert_fp8 ? 1.0 : 2.0;
    double kv = 0.0;
    for (int l = 0; l < c.n_layers; ++l)
      kv += (double)(is_full_layer(c, l) || c.window == 0 ? s->max_ctx : std::min(s->max_ctx, c.window));
    kv *= (double)s->max_batch * 2 * D.NKV * D.D * 2 / c.n_layers;
    const double attn = 2.0 * ((double)(D.NQ + 2 * D.NKV) * D.D * D.H + (double)D.H * D.NQ * D.D) + kv;
    const double moe = 2.0 * D.E * D.H + std::min(D.E, s->max_batch * D.K) * 3.0 * D.H * D.I * eb;
    a = (int)(n * attn / (attn + moe) + 0.5);
  }
  return std::max(D.NKV, std::min(a, n - 2));
}

static int build(mk_sched* s) {
  const mk_config& c = s->cfg;
  const ShapeDims& D = s->dims;
  const MoePlan& mp = s->plan;
  Builder B{s, s->max_batch, c.n_layers, D.E, D.NKV, D.K};
  const int MB = s->max_batch, L = c.n_layers, NKV = D.NKV, G = D.NQ / D.NKV;
  const int QKVROWS = (D.NQ + 2 * D.NKV) * D.D;
  const mk_sched_opts& o = s->opts;

  s->split_len = auto_split_pages(s) * c.page_size;
  const int full_slices = (s->max_ctx + s->split_len - 1) / s->split_len;
  s->n_static = 0;
  if (c.window > 0) {
    const int w_slices = (c.window + s->split_len - 1) / s->split_len + 1;
    s->n_static = std::min(full_slices, w_slices);
  }
  s->max_slots = std::max(full_slices, s->n_static);
  s->max_attn_entries = MB * NKV * full_slices;

  // tile sizes (multiples of the stage rows)
  const int sr_h = stage_rows(D.H), sr_o = stage_rows(G * D.D);
  auto round_to = [](int v, int m) { return std::max(m, (v / m) * m); };
  const int qkv_tile = o.qkv_tile_rows > 0 ? round_to(o.qkv_tile_rows, sr_h) : sr_h;
  if (D.D % qkv_tile != 0 || qkv_tile % sr_h != 0 || D.D % sr_h != 0)
    return fail(MK_ERR_ARG, "qkv_tile_rows must divide head_dim and be a multiple of the stage rows");
  const int o_tile = s->tc ? kTcDenseRows : o.o_tile_rows > 0 ? round_to(o.o_tile_rows, sr_o) : round_to(64, sr_o);
  // LM head: one tile per SM by default (the vocabulary split evenly in stage rows), so the
  // last wave of the step has no tail of SMs with one tile more than the others
  const int lm_even = ((c.vocab + s->num_sms - 1) / s->num_sms + sr_h - 1) / sr_h * sr_h;
  const int lm_tile = s->tc ? kTcDenseRows : o.lm_tile_rows > 0 ? round_to(o.lm_tile_rows, sr_h) : std::max(sr_h, lm_even);
  const int router_tile = s->tc ? std::min(kTcRouterRows, D.E) : sr_h * std::max(1, 16 / sr_h);
  // SMs of each branch: all of them, or the split of placement 2
  const int n_attn_sms = attn_group_sms(s), n_moe_sms = s->opts.placement == 2 ? s->num_sms - n_attn_sms : s->num_sms;
  const int n_moe = o.moe_claimers > 0 ? o.moe_claimers : n_moe_sms;
  const int attn_claim_default = std::min(n_attn_sms, std::max(1, MB * NKV * full_slices));
  const int n_attn = o.attn_claimers > 0 ? o.attn_claimers : attn_claim_default;
  // RMSNorm tasks: a row each for tcgen05 schedules (their rows run in parallel), else up to 4
  const int norm_rows = s->tc ? 1 : 4;

  B.alloc_layer_bars();
  std::vector<Desc> all;
  std::vector<size_t> layer_begin;  // first task of each layer (and of the final norm + LM head)

  for (int l = 0; l < L; ++l) {
    LayerBars& lb = s->lb[l];
    const bool full = is_full_layer(c, l);
    std::vector<Desc> w_norm = B.norm_wave(l, norm_rows);
    // one expert taken by every token: a dense SwiGLU FFN ("Tasks":
    // FFN_UPGATE_ACT, FFN_DOWN) in static tiles, with no routing
    const bool dense = D.E == 1 && D.K == 1;

    // QKV: a row tile never leaves one KV group's rows (its query heads, its
    // K head or its V head), so the group's attention waits on its own tiles
    std::vector<Desc> w_qkv;
    lb.n_qkv_g.assign(NKV, 0);
    const bool fuse_norm_qkv = o.fuse_norm_qkv && MB <= kTB;
    auto add_qkv = [&](int r0, int rows, int g) {
      Desc d = blank(OP_QKV_PROJ, l);
      d[F_A0] = r0;
      d[F_A0 + 1] = rows;
      if (fuse_norm_qkv) {  // the tile computes the RMSNorm: it waits for what the norm waits for
        d[F_WAIT0] = w_norm[0][F_WAIT0]; d[F_TGT0] = w_norm[0][F_TGT0];
        d[F_WAIT1] = w_norm[0][F_WAIT1]; d[F_TGT1] = w_norm[0][F_TGT1];
        d[F_A0 + 7] = 1;
      } else {
        B.wait(d, 0, lb.norm, lb.n_norm);
      }
      d[F_SIG0] = lb.qkv + g;
      lb.n_qkv_g[g]++;
      w_qkv.push_back(d);
    };
    if (s->tc) {
      // tcgen05 items: tiles of at most kTcDenseRows rows within each KV
      // group's query-head, K-head and V-head segments
      for (int g = 0; g < NKV; ++g) {
        const int seg_r0[3] = {g * G * D.D, (D.NQ + g) * D.D, (D.NQ + NKV + g) * D.D};
        const int seg_rows[3] = {G * D.D, D.D, D.D};
        for (int k = 0; k < 3; ++k)
          for (int r = 0; r < seg_rows[k]; r += kTcDenseRows)
            add_qkv(seg_r0[k] + r, std::min(kTcDenseRows, seg_rows[k] - r), g);
      }
    } else if (o.qkv_tile_rows > 0) {
      for (int r0 = 0; r0 < QKVROWS; r0 += qkv_tile) {
        const int head = r0 / D.D;
        add_qkv(r0, qkv_tile, head < D.NQ ? head / G : (head < D.NQ + NKV ? head - D.NQ : head - D.NQ - NKV));
      }
    } else {
      // one tile on each SM that holds none of the layer's routing tasks
      // (the RMSNorm, router and top-k tasks take the SMs just before the
      // tiles): each group segment gets tiles in proportion to its rows,
      // largest remainders first, as equal as the stage rows allow (full
      // shape: 142 tiles of 32 to 48 rows), so no SM holds two
      // every KV group gets the same tiles (its attention waits for a count
      // that is the same for all groups): a template of the group's three
      // segments -- query heads, K head, V head -- apportioned by largest
      // remainders, repeated per group
      struct Seg { int r0, rows, g, n; double frac; };
      const int n_routing = lb.n_norm + (dense ? 0 : (int)((D.E + router_tile - 1) / router_tile) +
                                                     (MB + kConsumerWarps - 1) / kConsumerWarps);
      const int per_group = std::max(3, (o.placement == 2 ? n_attn_sms : s->num_sms - n_routing) / NKV);
      Seg tmpl[3] = {{0, G * D.D, 0, 0, 0.0}, {0, D.D, 0, 0, 0.0}, {0, D.D, 0, 0, 0.0}};
      int given = 0;
      for (Seg& sg : tmpl) {
        const double share = (double)per_group * sg.rows / (G * D.D + 2 * D.D);
        sg.n = std::max(1, std::min((int)share, sg.rows / sr_h));
        sg.frac = share - (int)share;
        given += sg.n;
      }
      for (int pass = 0; pass < 3 && given < per_group; ++pass) {
        int best = -1;
        for (int k = 0; k < 3; ++k)
          if (tmpl[k].n < tmpl[k].rows / sr_h && (best < 0 || tmpl[k].frac > tmpl[best].frac)) best = k;
        if (best < 0) break;
        ++tmpl[best].n;
        tmpl[best].frac = -1.0;
        ++given;
      }
      std::vector<Seg> segs;
      for (int g = 0; g < NKV; ++g) {
        segs.push_back({g * G * D.D, G * D.D, g, tmpl[0].n, 0.0});
        segs.push_back({(D.NQ + g) * D.D, D.D, g, tmpl[1].n, 0.0});
        segs.push_back({(D.NQ + NKV + g) * D.D, D.D, g, tmpl[2].n, 0.0});
      }
      for (const Seg& sg : segs) {
        const int units = sg.rows / sr_h;
        const int n = sg.n;
        int r0 = sg.r0;
        for (int i = 0; i < n; ++i) {
          const int u = units / n + (i < units % n ? 1 : 0);
          add_qkv(r0, u * sr_h, sg.g);
          r0 += u * sr_h;
        }
      }
    }

    std::vector<Desc> w_router;
    if (!dense) w_router = B.dense_wave(OP_ROUTER_GEMM, l, D.E, router_tile, lb.router);
    lb.n_router = (int)w_router.size();
    const bool fuse_fin = o.fuse_finalize && MB <= kConsumerWarps;
    // routing fused into the router tasks: each counts itself in on lb.rarrive
    // and the last one runs the top-k and the queue build, then signals lb.fin;
    // at batch <= 2 each also computes the RMSNorm from the residual parts
    const bool fuse_rt = o.fuse_routing && fuse_fin;
    const bool norm_in_router = fuse_rt && MB <= kTB;
    for (size_t i = 0; i < w_router.size(); ++i) {
      Desc& d = w_router[i];
      if (norm_in_router) {
        d[F_WAIT0] = w_norm[0][F_WAIT0]; d[F_TGT0] = w_norm[0][F_TGT0];
        d[F_WAIT1] = w_norm[0][F_WAIT1]; d[F_TGT1] = w_norm[0][F_TGT1];
      } else {
        B.wait(d, 0, lb.norm, lb.n_norm);
      }
      if (fuse_rt) {
        d[F_A0 + 2] = lb.rarrive;
        d[F_A0 + 3] = lb.n_router;
        d[F_A0 + 4] = lb.fin;
        d[F_A0 + 5] = 1;
        d[F_A0 + 6] = (int)i;
        d[F_A0 + 7] = norm_in_router ? 1 : 0;
      }
    }

    std::vector<Desc> w_topk, w_fin;
    const int topk_rows = kConsumerWarps;
    for (int b0 = 0; b0 < (fuse_rt || dense ? 0 : MB); b0 += topk_rows) {
      Desc d = blank(OP_ROUTER_TOPK, l);
      d[F_A0] = b0;
      d[F_A0 + 1] = std::min(MB, b0 + topk_rows);
      d[F_A0 + 2] = fuse_fin ? 1 : 0;
      B.wait(d, 0, lb.router, lb.n_router);
      d[F_SIG0] = lb.topk;
      if (fuse_fin) d[F_SIG1] = lb.fin;
      w_topk.push_back(d);
    }
    lb.n_topk = (int)w_topk.size();
    if (!fuse_fin && !dense) {
      Desc d = blank(OP_ROUTE_FINALIZE, l);
      B.wait(d, 0, lb.topk, lb.n_topk);
      d[F_SIG0] = lb.fin;
      w_fin.push_back(d);
    }

    std::vector<Desc> w_gather;
    if (o.explicit_gather && !dense) {
      const int rows = MB * D.K, per = s->tc ? 8 : 32;  // tcgen05 schedules: more, smaller gathers
      for (int r0 = 0; r0 < rows; r0 += per) {
        Desc d = blank(OP_MOE_GATHER, l);
        d[F_A0] = r0;
        d[F_A0 + 1] = std::min(per, rows - r0);
        B.wait(d, 0, lb.fin, 1);
        if (norm_in_router) B.wait(d, 1, lb.norm, lb.n_norm);  // gathers the RMSNorm output
        d[F_SIG0] = lb.gather;
        w_gather.push_back(d);
      }
      lb.n_gather = (int)w_gather.size();
    }

    // attention: static slices for sliding layers, claimers for full layers
    std::vector<Desc> w_attn;
    if (full) {
      for (int i = 0; i < n_attn; ++i) {
        Desc d = blank(OP_ATTN_DRAIN, l);
        d[F_A0] = lb.claim_attn;
        d[F_A0 + 1] = lb.cnt;
        d[F_A0 + 2] = lb.qkv;
        d[F_A0 + 4] = o.attn_static ? i : -1;  // static: claimer i takes entries i, i + n, ...
        d[F_A0 + 5] = n_attn;
        d[F_SIG0] = lb.attn_done;
        w_attn.push_back(d);
      }
      lb.n_attn_claim = n_attn;
    } else {
      for (int b = 0; b < MB; ++b)
        for (int g = 0; g < NKV; ++g)
          for (int j = 0; j < s->n_static; ++j) {
            Desc d = blank(OP_ATTN_DECODE, l);
            d[F_A0] = b;
            d[F_A0 + 1] = g;
            d[F_A0 + 2] = j;
            d[F_A0 + 3] = lb.cnt;
            B.wait(d, 0, lb.qkv + g, lb.n_qkv_g[g]);
            d[F_SIG0] = lb.cnt + b * NKV + g;
            w_attn.push_back(d);
          }
    }
    // the QKV targets per group, for the drained slices
    for (auto& d : w_attn)
      if (d[F_OP] == OP_ATTN_DRAIN) d[F_A0 + 3] = lb.n_qkv_g[0];

    // one merge task per (row, group), or per (row, group, head) when there
    // are few rows: the merge is on the way from the last slice to the O tiles
    std::vector<Desc> w_acomb;
    lb.n_acomb_g.assign(NKV, 0);
    const int comb_heads = (o.combine_per_head && MB * NKV * G <= s->num_sms) ? G : 1;
    for (int b = 0; b < MB; ++b)
      for (int g = 0; g < NKV; ++g)
        for (int h = 0; h < comb_heads; ++h) {
          Desc d = blank(OP_ATTN_COMBINE, l);
          d[F_A0] = b;
          d[F_A0 + 1] = g;
          d[F_A0 + 2] = lb.cnt;
          d[F_A0 + 3] = comb_heads > 1 ? h : -1;
          B.wait(d, 0, lb.cnt + b * NKV + g, full ? TGT_DYN_SPLITS : s->n_static);
          d[F_SIG0] = lb.acomb + g;
          lb.n_acomb_g[g]++;
          w_acomb.push_back(d);
        }

    // MoE claimers: separate up/gate and down drains as on the pages (default),
    // or one queue of up/gate and down tiles with each expert's down tiles one
    // expert behind its up tiles (moe_queue = 1, slower: a down tile claimed
    // that early holds its SM's pipeline until the expert's up tiles land)
    std::vector<Desc> w_up, w_dn, w_mcomb;
    const bool unified = o.moe_queue == 1;
    if (dense) {
      // every up/gate tile reads the RMSNorm output; a down tile needs all
      // of the intermediate
      for (int t = 0; t < mp.up_tiles; ++t) {
        Desc d = blank(OP_FFN_UPGATE_ACT, l);
        d[F_A0] = t;
        B.wait(d, 0, lb.norm, lb.n_norm);
        d[F_SIG0] = lb.upd;
        w_up.push_back(d);
      }
      for (int t = 0; t < mp.dn_tiles; ++t) {
        Desc d = blank(OP_FFN_DOWN, l);
        d[F_A0] = t;
        B.wait(d, 0, lb.upd, mp.up_tiles);
        d[F_SIG0] = lb.dnd;
        w_dn.push_back(d);
      }
      lb.n_up_claim = mp.up_tiles;
      lb.n_dn_claim = mp.dn_tiles;
    }
    for (int i = 0; i < (dense ? 0 : n_moe); ++i) {
      Desc d = blank(OP_MOE_UPGATE_ACT_DRAIN, l);
      B.wait(d, 0, lb.fin, 1);
      // the routing can finish before the RMSNorm task when the routers
      // compute the norm themselves: the up/gate tiles read its output
      if (norm_in_router) B.wait(d, 1, lb.norm, lb.n_norm);
      d[F_A0] = lb.claim_up;
      d[F_A0 + 1] = lb.up;
      d[F_A0 + 2] = o.explicit_gather ? lb.gather : -1;
      d[F_A0 + 3] = o.explicit_gather ? lb.n_gather : 0;
      d[F_A0 + 4] = i;
      d[F_A0 + 5] = n_moe;
      d[F_A0 + 6] = unified ? 0 : 1;
      d[F_A0 + 7] = o.moe_static ? 1 : 0;
      d[F_SIG0] = unified ? lb.dnd : lb.upd;
      w_up.push_back(d);
      if (!unified) {
        Desc e = blank(OP_MOE_DOWN_DRAIN, l);
        B.wait(e, 0, lb.fin, 1);
        e[F_A0] = lb.claim_dn;
        e[F_A0 + 1] = lb.up;
        e[F_A0 + 2] = -1;
        e[F_A0 + 4] = i;
        e[F_A0 + 5] = n_moe;
        e[F_A0 + 7] = o.moe_static ? 1 : 0;
        e[F_SIG0] = lb.dnd;
        w_dn.push_back(e);
      }
    }
    if (!dense) lb.n_up_claim = lb.n_dn_claim = n_moe;
    if (!o.fuse_moe_combine) {
      for (int b0 = 0; b0 < MB; b0 += norm_rows) {
        Desc d = blank(OP_MOE_COMBINE, l);
        d[F_A0] = b0;
        d[F_A0 + 1] = std::min(MB, b0 + norm_rows);
        B.wait(d, 0, lb.dnd, lb.n_dn_claim);
        d[F_SIG0] = lb.mcomb;
        w_mcomb.push_back(d);
      }
      lb.n_mcomb = (int)w_mcomb.size();
    }

    std::vector<Desc> w_o;
    for (int r0 = 0; r0 < D.H; r0 += o_tile)
      for (int g = 0; g < NKV; ++g) {
        Desc d = blank(OP_O_PROJ, l);
        d[F_A0] = r0;
        d[F_A0 + 1] = std::min(o_tile, D.H - r0);
        d[F_A0 + 2] = g;
        B.wait(d, 0, lb.acomb + g, lb.n_acomb_g[g]);
        d[F_SIG0] = lb.o;
        w_o.push_back(d);
      }
    lb.n_o = (int)w_o.size();

    auto add = [&](std::vector<Desc>& w) { all.insert(all.end(), w.begin(), w.end()); };
    layer_begin.push_back(all.size());
    // the router and the routing head each layer's list: the MoE branch waits on
    // them, and QKV tiles would otherwise sit in front of them on their SMs
    add(w_norm);
    add(w_router);
    add(w_topk);
    add(w_fin);
    add(w_gather);
    add(w_qkv);
    switch (o.wave_order) {
      case MK_WAVES_INTERLEAVED:
        add(w_attn); add(w_up); add(w_dn); add(w_acomb); add(w_mcomb); add(w_o);
        break;
      case MK_WAVES_ATTN_FIRST:
        add(w_attn); add(w_acomb); add(w_o); add(w_up); add(w_dn); add(w_mcomb);
        break;
      case MK_WAVES_MOE_FIRST:
        add(w_up); add(w_attn); add(w_acomb); add(w_dn); add(w_o); add(w_mcomb);
        break;
      case MK_WAVES_MOE_FIRST_O:
        add(w_up); add(w_attn); add(w_acomb); add(w_o); add(w_dn); add(w_mcomb);
        break;
      case MK_WAVES_INTERLEAVED_O:
        add(w_attn); add(w_up); add(w_acomb); add(w_o); add(w_dn); add(w_mcomb);
        break;
      case MK_WAVES_O_BEFORE_DOWN:
        add(w_attn); add(w_acomb); add(w_up); add(w_o); add(w_dn); add(w_mcomb);
        break;
      default:
        add(w_attn); add(w_acomb); add(w_up); add(w_dn); add(w_o); add(w_mcomb);
        break;
    }
    if (o.moe_static && o.moe_balance && !unified && !dense && o.placement == 0)
      balance_moe_ranks(s, all, layer_begin.back(), MB, full);
  }
  // final RMSNorm and LM head
  std::vector<Desc> w_final = B.norm_wave(L, norm_rows);
  layer_begin.push_back(all.size());
  all.insert(all.end(), w_final.begin(), w_final.end());
  for (int r0 = 0; r0 < c.vocab; r0 += lm_tile) {
    Desc d = blank(OP_LM_HEAD, L);
    d[F_A0] = r0;
    d[F_A0 + 1] = std::min(lm_tile, c.vocab - r0);
    B.wait(d, 0, s->lb[L].norm, s->lb[L].n_norm);
    d[F_SIG0] = s->lm_bar;
    all.push_back(d);
  }

  // flatten: task k -> SM k mod #SMs, the greedy placement or the split
  const std::vector<int> sm_of = o.placement == 1   ? place_greedy(s, all, layer_begin, MB)
                                 : o.placement == 2 ? place_split(s, all, layer_begin, n_attn_sms)
                                 : o.placement == 3 ? place_affinity(s, all, layer_begin)
                                 : o.placement == 4 ? place_slices_free(s, all, layer_begin, MB, 3)
                                                    : std::vector<int>();
  s->tasks = std::move(all);
  s->per_sm.assign(s->num_sms, {});
  for (int k = 0; k < (int)s->tasks.size(); ++k) {
    s->tasks[k][F_TASK] = k;
    s->per_sm[o.placement != 0 ? sm_of[k] : k % s->num_sms].push_back(k);
  }
  return MK_OK;
}

static void layout_workspace(mk_sched* s) {
  const ShapeDims& D = s->dims;
  const int MB = s->max_batch, L = s->cfg.n_layers, G = D.NQ / D.NKV;
  WsLayout& w = s->ws;
  w = WsLayout();
  w.add("barriers", sizeof(uint32_t) * s->bar_kind.size());
  w.add("error", sizeof(uint32_t) * 8);
  w.add("progress", sizeof(uint32_t) * 8 * (size_t)s->num_sms);
  w.add("h", sizeof(float) * 2 * MB * D.H);  // the residual, by layer parity
  w.add("x", sizeof(float) * MB * D.H);
  w.add("q", sizeof(float) * MB * D.NQ * D.D);
  w.add("kvnew", 2ull * MB * 2 * D.NKV * D.D);
  w.add("part_o", sizeof(float) * (size_t)MB * D.NKV * s->max_slots * G * D.D);
  w.add("part_ml", sizeof(float) * (size_t)MB * D.NKV * s->max_slots * G * 2);
  w.add("attn_out", sizeof(float) * MB * D.NQ * D.D);
  w.add("opart", sizeof(float) * 2 * (size_t)D.NKV * MB * D.H);  // by layer parity
  w.add("router_logits", sizeof(float) * (size_t)L * MB * D.E);
  w.add("topk_ids", sizeof(int32_t) * (size_t)L * MB * D.K);
  w.add("topk_w", sizeof(float) * (size_t)L * MB * D.K);
  w.add("expert_count", sizeof(int32_t) * (size_t)L * D.E);
  w.add("expert_offset", sizeof(int32_t) * (D.E + 1));
  w.add("perm", sizeof(int32_t) * MB * D.K);
  w.add("inv", sizeof(int32_t) * MB * D.K);
  w.add("moe_queue", sizeof(int32_t) * 4 * (size_t)D.E);
  w.add("moe_queue_len", sizeof(int32_t) * 2);
  w.add("xg", s->opts.explicit_gather ? sizeof(float) * MB * D.K * D.H : 16);
  w.add("u", sizeof(float) * MB * D.K * D.I);
  w.add("y", sizeof(float) * (size_t)MB * D.K * D.H);
  w.add("moe_out", sizeof(float) * (size_t)MB * D.H);
  if (s->tc) {  // the BF16 hi/lo operand rows of the tcgen05 items (at least one box of rows each)
    w.add("xb", 2ull * s->tc_nb * D.H);
    w.add("attnb", 2ull * s->tc_nb * D.NQ * D.D);
    if (s->tc_fp8) {  // FP8 expert tiles: E4M3 term rows, one byte each, and the gathered rows' scales
      w.add("xg8", 1ull * std::max(kTcF8Terms * MB * D.K, s->tc_nb8) * D.H);
      w.add("xg8s", sizeof(float) * MB * D.K);
      w.add("u8", 1ull * std::max(kTcF8Terms * MB * D.K, s->tc_nb8) * D.I);
    } else {
      w.add("xgb", 2ull * std::max(2 * MB * D.K, s->tc_nb) * D.H);
      w.add("ub", 2ull * std::max(2 * MB * D.K, s->tc_nb) * D.I);
    }
  }
  if (s->opts.trace_hidden) w.add("hidden_trace", sizeof(float) * (size_t)(L + 1) * MB * D.H);
  if (s->opts.trace_queue) w.add("queue_trace", sizeof(int32_t) * (size_t)L * queue_trace_stride(D.E, MB * D.K));
  if (s->opts.trace) {
    size_t most = 0;
    for (const auto& l : s->per_sm) most = std::max(most, l.size());
    // tasks, plus the tiles and slices a claimer can take
    s->trace_cap = (int)(2 * most + 64 * (size_t)L + 1024);
    w.add("trace", sizeof(uint64_t) * 4 * (size_t)s->num_sms * s->trace_cap);
    w.add("stats", sizeof(uint64_t) * kStats * (size_t)s->num_sms);
  }
  w.total = (w.total + 255) & ~(size_t)255;
}

// ------------------------------------------------------------- validation

// Every barrier a task waits on must be fed by tasks that can run first, and
// a static barrier must receive exactly the count its waiters expect.  The
// lists are deadlock-free iff the graph of (list order on each SM) plus
// (producer -> barrier -> waiter) edges has no cycle.
static int validate(const mk_sched* s) {
  const int T = (int)s->tasks.size();
  const int NB = (int)s->bar_kind.size();
  std::vector<int> signals(NB, 0);
  std::vector<int> expect(NB, -1);
  std::vector<std::vector<int>> producers(NB), waiters(NB);
  auto add_wait = [&](int task, int bar, int tgt) {
    if (bar < 0) return 0;
    if (bar >= NB) return fail(MK_ERR_ARG, "task " + std::to_string(task) + " waits on barrier out of range");
    waiters[bar].push_back(task);
    if (s->bar_kind[bar] == BK_STATIC) {
      if (expect[bar] >= 0 && expect[bar] != tgt)
        return fail(MK_ERR_ARG, "barrier " + std::to_string(bar) + " waited on with two counts");
      expect[bar] = tgt;
    }
    return 0;
  };
  for (int t = 0; t < T; ++t) {
    const Desc& d = s->tasks[t];
    const int op = d[F_OP];
    if (op < 0 || op >= OP_COUNT) return fail(MK_ERR_ARG, "task " + std::to_string(t) + " has a bad opcode");
    for (int k : {F_SIG0, F_SIG1}) {
      const int b = d[k];
      if (b < 0) continue;
      if (b >= NB) return fail(MK_ERR_ARG, "task " + std::to_string(t) + " signals barrier out of range");
      signals[b]++;
      producers[b].push_back(t);
    }
    if (add_wait(t, d[F_WAIT0], d[F_TGT0]) || add_wait(t, d[F_WAIT1], d[F_TGT1])) return MK_ERR_ARG;
    // claimers: the tiles they run feed and wait on per-expert / per-row barriers
    // (a claimer of the combined queue both feeds and waits on the per-expert
    // counters; its queue order keeps every wait on earlier units, so only the
    // feeding edge enters the graph)
    if (op == OP_MOE_UPGATE_ACT_DRAIN)
      for (int e = 0; e < s->dims.E; ++e) producers[d[F_A0 + 1] + e].push_back(t);
    if (op == OP_MOE_DOWN_DRAIN)
      for (int e = 0; e < s->dims.E; ++e) waiters[d[F_A0 + 1] + e].push_back(t);
    if (op == OP_ATTN_DRAIN)
      for (int i = 0; i < s->max_batch * s->dims.NKV; ++i) producers[d[F_A0 + 1] + i].push_back(t);
    // fused routing: the last router task of the layer signals the routing
    // barrier once; every router task feeds it
    if (op == OP_ROUTER_GEMM && d[F_A0 + 5]) {
      const int b = d[F_A0 + 4];
      if (b < 0 || b >= NB) return fail(MK_ERR_ARG, "router task signals a barrier out of range");
      if (d[F_A0 + 6] == 0) signals[b]++;
      producers[b].push_back(t);
    }
  }
  for (int b = 0; b < NB; ++b) {
    if (s->bar_kind[b] != BK_STATIC) continue;
    if (expect[b] >= 0 && signals[b] != expect[b])
      return fail(MK_ERR_ARG, "barrier " + std::to_string(b) + " receives " + std::to_string(signals[b]) +
                                  " arrivals but is waited on for " + std::to_string(expect[b]));
  }
  // static slices of a sliding layer: the combine's count must equal the slices
  for (const Desc& d : s->tasks) {
    if (d[F_OP] != OP_ATTN_COMBINE || d[F_TGT0] == TGT_DYN_SPLITS) continue;
    const int b = d[F_WAIT0];
    int n = 0;
    for (int p : producers[b])
      if (s->tasks[p][F_OP] == OP_ATTN_DECODE) ++n;
    if (n != d[F_TGT0])
      return fail(MK_ERR_ARG, "attention counter " + std::to_string(b) + " gets " + std::to_string(n) +
                                  " slices, combine waits for " + std::to_string(d[F_TGT0]));
  }
  // cycle check (Kahn) over tasks and barriers
  const int N = T + NB;
  std::vector<std::vector<int>> adj(N);
  std::vector<int> indeg(N, 0);
  auto edge = [&](int a, int b) { adj[a].push_back(b); indeg[b]++; };
  for (const auto& lst : s->per_sm)
    for (size_t i = 1; i < lst.size(); ++i) edge(lst[i - 1], lst[i]);
  for (int b = 0; b < NB; ++b) {
    for (int p : producers[b]) edge(p, T + b);
    for (int w : waiters[b]) edge(T + b, w);
  }
  std::deque<int> q;
  for (int i = 0; i < N; ++i)
    if (indeg[i] == 0) q.push_back(i);
  int seen = 0;
  while (!q.empty()) {
    int v = q.front();
    q.pop_front();
    ++seen;
    for (int w : adj[v])
      if (--indeg[w] == 0) q.push_back(w);
  }
  if (seen != N) {
    for (int i = 0; i < T; ++i)
      if (indeg[i] > 0)
        return fail(MK_ERR_ARG, "cyclic wait: task " + std::to_string(i) + " (op " +
                                    std::to_string(s->tasks[i][F_OP]) + ", layer " +
                                    std::to_string(s->tasks[i][F_LAYER]) + ") can never start");
    return fail(MK_ERR_ARG, "cyclic wait between barriers");
  }
  // every waited barrier has at least one producer
  for (int b = 0; b < NB; ++b)
    if (!waiters[b].empty() && producers[b].empty() && s->bar_kind[b] != BK_CLAIM)
      return fail(MK_ERR_ARG, "barrier " + std::to_string(b) + " is waited on but never signalled");
  return MK_OK;
}

// ------------------------------------------------------------- simulation

namespace {

struct SimQueue {
  std::vector<int32_t> entries;
};

struct Sim {
  const mk_sched* s;
  int B;
  std::vector<int32_t> seq;
  std::vector<int32_t> routing;  // [L][B][K]
  std::vector<int64_t> bars;
  std::vector<int> pos;            // next task per SM
  std::vector<int> pending;        // claimed entry index per SM (-1 none)
  std::vector<int32_t> attn_q;
  std::vector<std::vector<int32_t>> up_q, dn_q, uni_q;  // per layer
  std::vector<int> first_done;  // per SM: the claimer's static first unit was taken
  std::vector<int64_t> last_unit;  // per SM: the claimer's current unit (static assignment)
  std::vector<int8_t> fin_done;
  std::string err;

  int64_t target(const Desc& d, int slot) {
    const int tgt = d[slot == 0 ? F_TGT0 : F_TGT1];
    if (tgt != TGT_DYN_SPLITS) return tgt;
    // combine of (b, g) in a full layer: the row's slice count (0 past the batch)
    const int b = d[F_A0];
    return b < B ? attn_slices(s, seq[b]) : 0;
  }

  bool waits_ok(const Desc& d) {
    for (int slot = 0; slot < 2; ++slot) {
      const int b = d[slot == 0 ? F_WAIT0 : F_WAIT1];
      if (b >= 0 && bars[b] < target(d, slot)) return false;
    }
    return true;
  }

  void signal(const Desc& d) {
    if (d[F_SIG0] >= 0) bars[d[F_SIG0]]++;
    if (d[F_SIG1] >= 0) bars[d[F_SIG1]]++;
  }

  // The layer's queues as the device derives them from the active-expert list:
  // entries (is_up, expert) for the combined queue, the up queue, the down queue.
  void finalize(int l) {
    const ShapeDims& D = s->dims;
    const int U = s->plan.up_tiles, DN = s->plan.dn_tiles;
    std::vector<int> count(D.E, 0), act;
    for (int b = 0; b < B; ++b)
      for (int j = 0; j < D.K; ++j) count[routing[((size_t)l * B + b) * D.K + j]]++;
    for (int e = 0; e < D.E; ++e)
      if (count[e]) act.push_back(e);
    const int n = (int)act.size();
    up_q[l].clear();
    dn_q[l].clear();
    uni_q[l].clear();
    for (int a = 0; a < n; ++a) {
      for (int t = 0; t < U; ++t) up_q[l].push_back(act[a]);
      for (int t = 0; t < DN; ++t) dn_q[l].push_back(act[a]);
    }
    for (int t = 0; t < U; ++t) uni_q[l].push_back(act[0] | (1 << 30));
    for (int a = 1; a < n; ++a) {
      for (int t = 0; t < U; ++t) uni_q[l].push_back(act[a] | (1 << 30));
      for (int t = 0; t < DN; ++t) uni_q[l].push_back(act[a - 1]);
    }
    for (int t = 0; t < DN; ++t) uni_q[l].push_back(act[n - 1]);
    fin_done[l] = 1;
  }

  // One step of SM `sm`; returns true if it made progress.
  bool step(int sm) {
    const auto& lst = s->per_sm[sm];
    if (pos[sm] >= (int)lst.size()) return false;
    const Desc& d = s->tasks[lst[pos[sm]]];
    const int op = d[F_OP], l = d[F_LAYER];
    const int NKV = s->dims.NKV;
    if (!waits_ok(d)) return false;
    switch (op) {
      case OP_ROUTER_TOPK:
        if (d[F_A0 + 2]) finalize(l);
        signal(d);
        break;
      case OP_ROUTER_GEMM:
        signal(d);
        if (d[F_A0 + 5] && ++bars[d[F_A0 + 2]] == d[F_A0 + 3]) {  // the last router task
          finalize(l);
          bars[d[F_A0 + 4]]++;
        }
        break;
      case OP_ROUTE_FINALIZE:
        finalize(l);
        signal(d);
        break;
      case OP_ATTN_DRAIN: {
        const int claim = d[F_A0];
        if (pending[sm] < 0) {
          int64_t i;
          if (d[F_A0 + 4] >= 0) {  // static: entries i, i + n, ...
            i = first_done[sm] ? last_unit[sm] + d[F_A0 + 5] : d[F_A0 + 4];
            first_done[sm] = 1;
            last_unit[sm] = i;
          } else {
            i = bars[claim]++;
          }
          if (i >= (int64_t)attn_q.size()) {
            first_done[sm] = 0;
            signal(d);
            break;
          }
          pending[sm] = (int)i;
        }
        const int32_t e = attn_q[pending[sm]];
        const int b = (e >> 24) & 0xff, g = (e >> 20) & 0xf;
        if (bars[d[F_A0 + 2] + g] < d[F_A0 + 3]) return false;  // QKV of this group not done
        bars[d[F_A0 + 1] + b * NKV + g]++;
        pending[sm] = -1;
        return true;  // the claimer stays on this task
      }
      case OP_MOE_UPGATE_ACT_DRAIN:
      case OP_MOE_DOWN_DRAIN: {
        if (!fin_done[l]) {
          err = "MoE claimer ran before its queue was built (layer " + std::to_string(l) + ")";
          return false;
        }
        const int mode = op == OP_MOE_DOWN_DRAIN ? 2 : d[F_A0 + 6];
        auto& q = mode == 0 ? uni_q[l] : mode == 1 ? up_q[l] : dn_q[l];
        const int claim = d[F_A0];
        if (pending[sm] < 0) {
          // the first unit is the claimer's own index; later ones come from the counter
          int64_t i;
          const int64_t n = d[F_A0 + 5];
          if (!first_done[sm]) {
            i = d[F_A0 + 4];
            // static down units start where the up units left off, so the
            // claimers with an extra up/gate tile get no extra down tile
            if (d[F_A0 + 7] == 1 && mode == 2) i = (i + n - (int64_t)up_q[l].size() % n) % n;
            first_done[sm] = 1;
          } else {
            i = d[F_A0 + 7] ? last_unit[sm] + n : n + bars[claim]++;
          }
          last_unit[sm] = i;
          if (i >= (int64_t)q.size()) {
            first_done[sm] = 0;
            signal(d);
            break;
          }
          pending[sm] = (int)i;
        }
        const int32_t u = q[pending[sm]];
        const bool up = mode == 1 || (mode == 0 && (u & (1 << 30)));
        const int e = u & 0xffff;
        if (up) {
          if (d[F_A0 + 2] >= 0 && bars[d[F_A0 + 2]] < d[F_A0 + 3]) return false;
          bars[d[F_A0 + 1] + e]++;
        } else {
          if (bars[d[F_A0 + 1] + e] < s->plan.up_tiles) return false;  // up tiles of e not done
        }
        pending[sm] = -1;
        return true;
      }
      default:
        signal(d);
        break;
    }
    pos[sm]++;
    return true;
  }
};

}  // namespace

static void build_attn_queue(const mk_sched* s, int B, const int32_t* seq, std::vector<int32_t>& q) {
  q.clear();
  for (int b = 0; b < B; ++b)
    for (int g = 0; g < s->dims.NKV; ++g)
      for (int j = 0; j < attn_slices(s, seq[b]); ++j) q.push_back((b << 24) | (g << 20) | j);
}

}  // namespace mk

using namespace mk;

// The tensor-core schedules' default wave order: there most expert tiles
// are GEMV or tcgen05 items that can stream while the attention slices wait
// for their queries, so the MoE waves go right behind the slices (ragged
// batch 32: 9.82 ms interleaved against 10.03 with O-proj before the down
// tiles and 12.0 in the batch-1 order); up to 8 rows, where the merges and
// O-proj tiles are few and short, O-proj before the down tiles (batch 4:
// 4.07 against 4.16 ms interleaved).
int tc_wave_order(int max_batch) {
  return max_batch <= 8 ? MK_WAVES_O_BEFORE_DOWN : MK_WAVES_INTERLEAVED;
}

extern "C" {

void mk_default_sched_opts(mk_sched_opts* o) {
  std::memset(o, 0, sizeof(*o));
  o->wave_order = -1;
  o->fuse_finalize = 1;
  o->fuse_moe_combine = 1;
  o->moe_static = -1;
  o->fuse_routing = 1;
  o->fuse_norm_qkv = 1;
  o->attn_static = 1;
  o->moe_balance = 0;
  o->combine_per_head = 0;
  o->placement = 0;
}

int mk_build_tasks(const mk_model* m, int32_t max_batch, int32_t max_ctx, const mk_sched_opts* opts,
                   mk_sched** out) {
  if (!m || !out) return fail(MK_ERR_ARG, "null argument");
  *out = nullptr;
  if (max_batch < 1 || max_batch > kMaxBatch) return fail(MK_ERR_ARG, "max_batch must be in [1, 64]");
  if (max_ctx < 1) return fail(MK_ERR_ARG, "max_ctx must be >= 1");
  if (m->cfg.expert_fp4 && max_batch > kTB) return fail(MK_ERR_UNSUPPORTED, "FP4 experts are compiled for max_batch <= 2");
  if (m->cfg.expert_fp8 && max_batch > kTcF8MaxBatch)
    return fail(MK_ERR_UNSUPPORTED, "FP8 experts are compiled for max_batch <= " + std::to_string(kTcF8MaxBatch) +
                                        " (the MMA's N holds four E4M3 term rows per routed row)");
  if (m->cfg.expert_fp8 && max_batch > kTB && (m->dims.H % kTcK8 || m->dims.I % kTcK8))
    return fail(MK_ERR_UNSUPPORTED, "FP8 experts above batch 2 need hidden and inter multiples of 128");
  mk_sched* s = new mk_sched();
  s->cfg = m->cfg;
  s->dims = m->dims;
  s->plan = m->plan;
  if (opts) s->opts = *opts;
  else mk_default_sched_opts(&s->opts);
  s->max_batch = max_batch;
  s->max_ctx = max_ctx;
  // batches beyond the GEMV's kTB rows: the weight tiles are real contractions,
  // run on the tcgen05 tensor cores (BF16 or FP8 experts of an MoE model)
  // (FP8 experts: the expert tiles on FP8 MMAs against E4M3 term rows)
  s->tc = max_batch > kTB && !m->cfg.expert_fp4 && !(m->dims.E == 1 && m->dims.K == 1);
  if (s->tc) {
    s->tc_fp8 = m->cfg.expert_fp8 != 0;
    s->plan = s->tc_fp8 ? moe_plan_tc8(m->dims) : moe_plan_tc(m->dims);
    s->tc_nb = (2 * max_batch + 15) / 16 * 16;
    s->tc_nb8 = s->tc_fp8 ? (kTcF8Terms * max_batch + 15) / 16 * 16 : 0;
    s->opts.explicit_gather = 1;  // the up/gate tiles take their rows in expert order
  }
  // MoE claims: static for the GEMV builds (their tiles are short and equal),
  // dynamic for tensor-core schedules (long tiles whose count rarely divides
  // the claimers: the SMs that finish first take the rest)
  if (s->opts.moe_static < 0) s->opts.moe_static = s->tc ? 0 : 1;
  s->num_sms = s->opts.num_sms;
  if (s->num_sms <= 0) {
    s->num_sms = query_num_sms();
    if (s->num_sms <= 0) {
      delete s;
      return fail(MK_ERR_CUDA, "cannot query the SM count (no device?); pass opts.num_sms");
    }
  }
  if (s->opts.wave_order == -1) s->opts.wave_order = s->tc ? tc_wave_order(max_batch) : MK_WAVES_DEFAULT;
  if (s->opts.wave_order < 0 || s->opts.wave_order > 6) {
    delete s;
    return fail(MK_ERR_ARG, "unknown wave order");
  }
  if (s->opts.placement < 0 || s->opts.placement > 4) {
    delete s;
    return fail(MK_ERR_ARG, "unknown placement");
  }
  s->watchdog_ns = (int64_t)(s->opts.watchdog_ms > 0 ? s->opts.watchdog_ms : 2000) * 1000000;
  int rc = build(s);
  if (rc == MK_OK) rc = validate(s);
  if (rc != MK_OK) {
    delete s;
    return rc;
  }
  s->lean = true;
  for (const Desc& d : s->tasks) {
    const int op = d[F_OP];
    if (op == OP_ROUTER_TOPK || op == OP_ROUTE_FINALIZE || op == OP_MOE_GATHER || op == OP_MOE_COMBINE ||
        (op == OP_ATTN_COMBINE && d[F_A0 + 3] >= 0) || (op == OP_ATTN_DRAIN && d[F_A0 + 4] < 0) ||
        (op == OP_MOE_UPGATE_ACT_DRAIN && (d[F_A0 + 6] != 1 || d[F_A0 + 7] == 0)) ||
        (op == OP_MOE_DOWN_DRAIN && d[F_A0 + 7] == 0))
      s->lean = false;
  }
  layout_workspace(s);
  *out = s;
  return MK_OK;
}

void mk_free_sched(mk_sched* s) { delete s; }

size_t mk_sched_bytes(const mk_sched* s) {
  if (!s) return 0;
  return sizeof(int32_t) * (2 * (size_t)s->num_sms + 32 * s->tasks.size()) + 128;
}

size_t mk_workspace_bytes(const mk_sched* s) { return s ? s->ws.total : 0; }

int64_t mk_workspace_offset(const mk_sched* s, const char* name) {
  if (!s || !name) return -1;
  if (!std::strcmp(name, "moe_queue_len")) return (int64_t)s->ws.off("moe_queue_len");
  const size_t o = s->ws.off(name);
  return o == (size_t)-1 ? -1 : (int64_t)o;
}

int32_t mk_sched_num_sms(const mk_sched* s) { return s ? s->num_sms : 0; }

int32_t mk_sched_num_tasks(const mk_sched* s, int32_t sm) {
  if (!s || sm < 0 || sm >= s->num_sms) return -1;
  return (int32_t)s->per_sm[sm].size();
}

int32_t mk_sched_num_barriers(const mk_sched* s) { return s ? (int32_t)s->bar_kind.size() : 0; }

int mk_sched_get_task(const mk_sched* s, int32_t sm, int32_t idx, int32_t desc[32]) {
  if (!s || sm < 0 || sm >= s->num_sms || idx < 0 || idx >= (int)s->per_sm[sm].size() || !desc)
    return fail(MK_ERR_ARG, "task index out of range");
  std::memcpy(desc, s->tasks[s->per_sm[sm][idx]].data(), sizeof(int32_t) * 32);
  return MK_OK;
}

int mk_sched_set_task(mk_sched* s, int32_t sm, int32_t idx, const int32_t desc[32]) {
  if (!s || sm < 0 || sm >= s->num_sms || idx < 0 || idx >= (int)s->per_sm[sm].size() || !desc)
    return fail(MK_ERR_ARG, "task index out of range");
  std::memcpy(s->tasks[s->per_sm[sm][idx]].data(), desc, sizeof(int32_t) * 32);
  return MK_OK;
}

int mk_sched_validate(const mk_sched* s) {
  if (!s) return fail(MK_ERR_ARG, "null schedule");
  return validate(s);
}

int mk_sched_simulate(const mk_sched* s, int32_t batch, const int32_t* seq_lens,
                      const int32_t* routing, uint64_t seed) {
  if (!s || !seq_lens || batch < 1 || batch > s->max_batch) return fail(MK_ERR_ARG, "bad batch");
  const int L = s->cfg.n_layers, K = s->dims.K, E = s->dims.E;
  Sim sim;
  sim.s = s;
  sim.B = batch;
  sim.seq.assign(seq_lens, seq_lens + batch);
  for (int b = 0; b < batch; ++b)
    if (seq_lens[b] < 1 || seq_lens[b] > s->max_ctx) return fail(MK_ERR_ARG, "seq_len out of range");
  std::mt19937_64 rng(seed);
  sim.routing.resize((size_t)L * batch * K);
  for (int l = 0; l < L; ++l)
    for (int b = 0; b < batch; ++b) {
      int32_t* r = &sim.routing[((size_t)l * batch + b) * K];
      if (routing) {
        std::memcpy(r, routing + ((size_t)l * batch + b) * K, sizeof(int32_t) * K);
      } else {
        std::vector<int> ex(E);
        for (int e = 0; e < E; ++e) ex[e] = e;
        std::shuffle(ex.begin(), ex.end(), rng);
        for (int j = 0; j < K; ++j) r[j] = ex[j];
      }
    }
  sim.bars.assign(s->bar_kind.size(), 0);
  sim.pos.assign(s->num_sms, 0);
  sim.pending.assign(s->num_sms, -1);
  build_attn_queue(s, batch, seq_lens, sim.attn_q);
  sim.up_q.assign(L, {});
  sim.dn_q.assign(L, {});
  sim.uni_q.assign(L, {});
  sim.first_done.assign(s->num_sms, 0);
  sim.last_unit.assign(s->num_sms, 0);
  sim.fin_done.assign(L, 0);
  std::vector<int> order(s->num_sms);
  for (int i = 0; i < s->num_sms; ++i) order[i] = i;
  for (;;) {
    std::shuffle(order.begin(), order.end(), rng);
    bool progress = false;
    for (int sm : order) progress |= sim.step(sm);
    if (!sim.err.empty()) return fail(MK_ERR_ARG, sim.err);
    if (!progress) break;
  }
  {
    // a deadlock: report the stuck SMs of the earliest layer with what they wait on
    std::string msg;
    int n = 0, min_layer = 1 << 30;
    for (int sm = 0; sm < s->num_sms; ++sm)
      if (sim.pos[sm] < (int)s->per_sm[sm].size())
        min_layer = std::min(min_layer, (int)s->tasks[s->per_sm[sm][sim.pos[sm]]][F_LAYER]);
    std::map<int, int> hist;
    for (int sm = 0; sm < s->num_sms; ++sm)
      if (sim.pos[sm] < (int)s->per_sm[sm].size()) hist[s->tasks[s->per_sm[sm][sim.pos[sm]]][F_OP] * 100 + s->tasks[s->per_sm[sm][sim.pos[sm]]][F_LAYER]]++;
    for (auto& kv : hist) msg += "[op " + std::to_string(kv.first / 100) + " layer " + std::to_string(kv.first % 100) + ": " + std::to_string(kv.second) + " SMs] ";
    for (int sm = 0; sm < s->num_sms && n < 4; ++sm)
      if (sim.pos[sm] < (int)s->per_sm[sm].size()) {
        const Desc& d = s->tasks[s->per_sm[sm][sim.pos[sm]]];
        if (d[F_LAYER] != min_layer) continue;
        msg += (n++ ? "; " : "") + std::string("SM ") + std::to_string(sm) + " stuck at task " +
               std::to_string(d[F_TASK]) + " (op " + std::to_string(d[F_OP]) + ", layer " +
               std::to_string(d[F_LAYER]) + ", waits " + std::to_string(d[F_WAIT0]) + ":" +
               std::to_string(d[F_WAIT0] >= 0 ? sim.bars[d[F_WAIT0]] : 0) + "/" + std::to_string(sim.target(d, 0)) +
               (sim.pending[sm] >= 0 ? ", unit " + std::to_string(sim.pending[sm]) : std::string()) + ")";
      }
    if (n) return fail(MK_ERR_ARG, "deadlock: " + msg);
  }
  // every static barrier ends at exactly the count its waiters expect
  std::vector<int64_t> expect(s->bar_kind.size(), -1);
  for (const Desc& d : s->tasks)
    for (int slot = 0; slot < 2; ++slot) {
      const int b = d[slot == 0 ? F_WAIT0 : F_WAIT1];
      if (b >= 0 && s->bar_kind[b] == BK_STATIC) expect[b] = d[slot == 0 ? F_TGT0 : F_TGT1];
    }
  for (size_t b = 0; b < expect.size(); ++b)
    if (expect[b] >= 0 && sim.bars[b] != expect[b])
      return fail(MK_ERR_ARG, "barrier " + std::to_string(b) + " ended at " + std::to_string(sim.bars[b]) +
                                  ", expected " + std::to_string(expect[b]));
  // attention counters: each row's slices, each expert's up tiles
  for (int l = 0; l < L; ++l) {
    const LayerBars& lb = s->lb[l];
    for (int b = 0; b < s->max_batch; ++b)
      for (int g = 0; g < s->dims.NKV; ++g) {
        const int64_t want = b >= batch ? (is_full_layer(s->cfg, l) ? 0 : s->n_static)
                                        : (is_full_layer(s->cfg, l) ? attn_slices(s, seq_lens[b]) : s->n_static);
        if (sim.bars[lb.cnt + b * s->dims.NKV + g] != want)
          return fail(MK_ERR_ARG, "attention counter of layer " + std::to_string(l) + " row " +
                                      std::to_string(b) + " ended at " +
                                      std::to_string(sim.bars[lb.cnt + b * s->dims.NKV + g]));
      }
  }
  return MK_OK;
}

}  // extern "C"
