// Token-budget packer: builds the mixed batch descriptor for one step.
//
// Priority order from the pofe.ai "Chunked prefill" page ("How it works, step
// by step", steps 1-3): decodes, then partial prefills, then admissions.  The
// readings taken where the pages are silent or disagree are listed beside
// mb_sched_create in include/mb.h.  Host only; no device work.

#include <cstdint>
#include <algorithm>
#include <cstring>
#include <deque>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "mb.h"
#include "mb_internal.h"

namespace {

constexpr int32_t kPage = MB_PAGE_TOKENS;

inline int32_t pages_for(int64_t tokens) { return static_cast<int32_t>((tokens + kPage - 1) / kPage); }

struct Req {
  int64_t id;
  int32_t prompt_len;
  int64_t computed;           // tokens in the KV cache
  std::vector<int32_t> pages; // block table
  int state;                  // 0 waiting, 1 partial, 2 running
};

}  // namespace

struct mb_sched {
  mb_pack_cfg cfg;
  int32_t num_pages;
  // adaptive per-step chunk cap (mb_sched_set_adaptive); ad_min == 0: off
  int32_t ad_min = 0, ad_base = 0, ad_max = 0, ad_pressure = 0;
  std::deque<int32_t> free_pages;
  std::unordered_map<int64_t, Req *> by_id;
  // Queues hold pointers into by_id's objects; std::list keeps FIFO order with
  // O(1) removal of a known element.
  std::list<Req *> running, partial, waiting;
  // output arrays of the last pack
  std::vector<int32_t> qo_indptr, kv_len, bt_indptr, bt;
  std::vector<int64_t> ids;

  ~mb_sched() {
    for (auto &kv : by_id) delete kv.second;
  }

  void take(Req *r, int32_t n) {
    for (int32_t i = 0; i < n; ++i) {
      r->pages.push_back(free_pages.front());
      free_pages.pop_front();
    }
  }
};

extern "C" {

mb_status mb_sched_create(const mb_pack_cfg *cfg, int32_t num_pages, const int32_t *free_order,
                          mb_sched **out) {
  if (!cfg || !out || num_pages < 0 || (num_pages > 0 && !free_order))
    return mb::fail(MB_EINVAL, "mb_sched_create: null argument or negative page count");
  if (cfg->budget < 1 || cfg->max_seqs < 1 || cfg->chunk_cap < 0)
    return mb::fail(MB_EINVAL, "mb_sched_create: budget and max_seqs must be >= 1, chunk_cap >= 0");
  std::vector<char> seen(static_cast<size_t>(num_pages), 0);
  for (int32_t i = 0; i < num_pages; ++i) {
    int32_t p = free_order[i];
    if (p < 0 || p >= num_pages || seen[p])
      return mb::fail(MB_EINVAL, "mb_sched_create: free_order is not a permutation of 0..num_pages-1");
    seen[p] = 1;
  }
  mb_sched *s = new (std::nothrow) mb_sched();
  if (!s) return mb::fail(MB_ENOMEM, "mb_sched_create: out of host memory");
  s->cfg = *cfg;
  s->num_pages = num_pages;
  s->free_pages.assign(free_order, free_order + num_pages);
  *out = s;
  return MB_OK;
}

mb_status mb_sched_add(mb_sched *s, int64_t req_id, int32_t prompt_len, int32_t computed) {
  if (!s) return mb::fail(MB_EINVAL, "mb_sched_add: null scheduler");
  if (prompt_len < 1 || computed < 0)
    return mb::fail(MB_EINVAL, "mb_sched_add: prompt_len must be >= 1 and computed >= 0");
  if (s->by_id.count(req_id)) return mb::fail(MB_EINVAL, "mb_sched_add: duplicate request id");
  int32_t need = pages_for(computed);
  if (need > static_cast<int64_t>(s->free_pages.size()))
    return mb::fail(MB_ENOSPACE, "mb_sched_add: not enough free pages for the cached tokens");
  Req *r = new (std::nothrow) Req{req_id, prompt_len, computed, {}, 0};
  if (!r) return mb::fail(MB_ENOMEM, "mb_sched_add: out of host memory");
  s->take(r, need);
  s->by_id[req_id] = r;
  if (computed == 0) {
    r->state = 0;
    s->waiting.push_back(r);
  } else if (computed < prompt_len) {
    r->state = 1;
    s->partial.push_back(r);
  } else {
    r->state = 2;
    s->running.push_back(r);
  }
  return MB_OK;
}

mb_status mb_sched_finish(mb_sched *s, int64_t req_id) {
  if (!s) return mb::fail(MB_EINVAL, "mb_sched_finish: null scheduler");
  auto it = s->by_id.find(req_id);
  if (it == s->by_id.end()) return mb::fail(MB_EINVAL, "mb_sched_finish: unknown request id");
  Req *r = it->second;
  std::list<Req *> &q = r->state == 0 ? s->waiting : (r->state == 1 ? s->partial : s->running);
  q.remove(r);
  for (int32_t p : r->pages) s->free_pages.push_back(p);
  s->by_id.erase(it);
  delete r;
  return MB_OK;
}

mb_status mb_sched_pack(mb_sched *s, mb_sched_batch *out) {
  if (!s || !out) return mb::fail(MB_EINVAL, "mb_sched_pack: null argument");
  struct Row {
    Req *r;
    int32_t n;
    bool prefill;
  };
  std::vector<Row> rows;
  int64_t left = s->cfg.budget;
  int64_t cap = s->cfg.chunk_cap;
  if (s->ad_min > 0) {
    // this step's chunk size from the decode load (llm-stack-book 7.8,
    // "Priority and Preemption Policies", adaptive_chunk_size): the largest
    // chunks with no decode running, the smallest from `pressure` decodes
    // on, linearly from base down to min in between (truncated)
    const int64_t depth = static_cast<int64_t>(s->running.size());
    int64_t eff;
    if (depth == 0) {
      eff = s->ad_max;
    } else if (depth >= s->ad_pressure) {
      eff = s->ad_min;
    } else {
      const double ratio = static_cast<double>(depth) / static_cast<double>(s->ad_pressure);
      eff = static_cast<int64_t>(static_cast<double>(s->ad_base) - ratio * static_cast<double>(s->ad_base - s->ad_min));
      eff = std::max<int64_t>(s->ad_min, std::min<int64_t>(eff, s->ad_base));
    }
    cap = cap ? std::min(cap, eff) : eff;
  }

  // 1. one token per running decode, while a budget unit is left
  for (Req *r : s->running) {
    if (left < 1) break;
    int32_t need = pages_for(r->computed + 1) - static_cast<int32_t>(r->pages.size());
    if (need > static_cast<int64_t>(s->free_pages.size())) continue;  // no page: skipped this step
    s->take(r, need);
    rows.push_back({r, 1, false});
    left -= 1;
  }
  // 2. next chunk of every partial prefill, FIFO
  for (Req *r : s->partial) {
    if (left <= 0) break;
    int64_t n = std::min<int64_t>(left, r->prompt_len - r->computed);
    if (cap) n = std::min(n, cap);
    int64_t room = (static_cast<int64_t>(r->pages.size()) + static_cast<int64_t>(s->free_pages.size())) * kPage -
                   r->computed;
    n = std::min(n, room);
    if (n <= 0) continue;
    s->take(r, pages_for(r->computed + n) - static_cast<int32_t>(r->pages.size()));
    rows.push_back({r, static_cast<int32_t>(n), true});
    left -= n;
  }
  // 3. admissions in arrival order; stop at the first refusal
  while (!s->waiting.empty() && left > 0) {
    Req *r = s->waiting.front();
    if (static_cast<int64_t>(s->running.size() + s->partial.size()) >= s->cfg.max_seqs) break;
    int64_t n = std::min<int64_t>(left, r->prompt_len);
    if (cap) n = std::min(n, cap);
    if (pages_for(n) > static_cast<int64_t>(s->free_pages.size())) break;
    s->waiting.pop_front();
    r->state = 1;
    s->partial.push_back(r);
    s->take(r, pages_for(n));
    rows.push_back({r, static_cast<int32_t>(n), true});
    left -= n;
  }

  // emit CSR and advance the state as if the pass ran
  s->qo_indptr.assign(1, 0);
  s->bt_indptr.assign(1, 0);
  s->kv_len.clear();
  s->bt.clear();
  s->ids.clear();
  for (const Row &row : rows) {
    Req *r = row.r;
    r->computed += row.n;
    s->qo_indptr.push_back(s->qo_indptr.back() + row.n);
    s->kv_len.push_back(static_cast<int32_t>(r->computed));
    s->bt.insert(s->bt.end(), r->pages.begin(), r->pages.end());
    s->bt_indptr.push_back(static_cast<int32_t>(s->bt.size()));
    s->ids.push_back(r->id);
    if (row.prefill && r->computed >= r->prompt_len) {
      s->partial.remove(r);
      r->state = 2;
      s->running.push_back(r);
    }
  }
  out->batch.num_reqs = static_cast<int32_t>(rows.size());
  out->batch.qo_indptr = s->qo_indptr.data();
  out->batch.kv_len = s->kv_len.data();
  out->batch.bt_indptr = s->bt_indptr.data();
  out->batch.bt = s->bt.data();
  out->req_ids = s->ids.data();
  return MB_OK;
}

mb_status mb_sched_set_adaptive(mb_sched *s, int32_t min_chunk, int32_t base_chunk, int32_t max_chunk,
                                int32_t decode_pressure) {
  if (!s) return mb::fail(MB_EINVAL, "mb_sched_set_adaptive: null scheduler");
  if (min_chunk == 0) {
    s->ad_min = s->ad_base = s->ad_max = s->ad_pressure = 0;
    return MB_OK;
  }
  if (min_chunk < 1 || base_chunk < min_chunk || max_chunk < base_chunk || decode_pressure < 1)
    return mb::fail(MB_EINVAL, "mb_sched_set_adaptive: need 1 <= min <= base <= max and decode_pressure >= 1");
  s->ad_min = min_chunk;
  s->ad_base = base_chunk;
  s->ad_max = max_chunk;
  s->ad_pressure = decode_pressure;
  return MB_OK;
}

mb_status mb_sched_counts(const mb_sched *s, int32_t counts[4]) {
  if (!s || !counts) return mb::fail(MB_EINVAL, "mb_sched_counts: null argument");
  counts[0] = static_cast<int32_t>(s->free_pages.size());
  counts[1] = static_cast<int32_t>(s->running.size());
  counts[2] = static_cast<int32_t>(s->partial.size());
  counts[3] = static_cast<int32_t>(s->waiting.size());
  return MB_OK;
}

mb_status mb_sched_destroy(mb_sched *s) {
  delete s;
  return MB_OK;
}

}  // extern "C"
