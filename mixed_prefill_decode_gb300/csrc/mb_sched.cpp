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

// checkpoint words: magic, version, then budget, max_seqs, chunk_cap,
// num_pages, the four adaptive settings and the free-list length
constexpr int64_t kStateMagic = 0x4D4253434844;   // "MBSCHD"
constexpr int64_t kStateVersion = 1;
constexpr int64_t kStateHeaderWords = 11;

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

// ---------------------------------------------------------------- checkpoint
// The packer's whole state as int64 words (layout in include/mb.h beside
// mb_sched_save).  Queue and free-list order are kept: they decide every
// later batch.

mb_status mb_sched_save(const mb_sched *s, int64_t *buf, int64_t cap, int64_t *len) {
  if (!s || !len || cap < 0 || (cap > 0 && !buf)) return mb::fail(MB_EINVAL, "mb_sched_save: null argument");
  int64_t need = kStateHeaderWords + static_cast<int64_t>(s->free_pages.size()) + 3;
  for (const std::list<Req *> *q : {&s->running, &s->partial, &s->waiting})
    for (const Req *r : *q) need += 4 + static_cast<int64_t>(r->pages.size());
  *len = need;
  if (!buf) return MB_OK;
  if (cap < need)
    return mb::fail(MB_ENOSPACE, "mb_sched_save: buffer holds %lld words, the state needs %lld",
                    static_cast<long long>(cap), static_cast<long long>(need));
  int64_t *w = buf;
  *w++ = kStateMagic;
  *w++ = kStateVersion;
  *w++ = s->cfg.budget;
  *w++ = s->cfg.max_seqs;
  *w++ = s->cfg.chunk_cap;
  *w++ = s->num_pages;
  *w++ = s->ad_min;
  *w++ = s->ad_base;
  *w++ = s->ad_max;
  *w++ = s->ad_pressure;
  *w++ = static_cast<int64_t>(s->free_pages.size());
  for (int32_t p : s->free_pages) *w++ = p;
  for (const std::list<Req *> *q : {&s->running, &s->partial, &s->waiting}) {
    *w++ = static_cast<int64_t>(q->size());
    for (const Req *r : *q) {
      *w++ = r->id;
      *w++ = r->prompt_len;
      *w++ = r->computed;
      *w++ = static_cast<int64_t>(r->pages.size());
      for (int32_t p : r->pages) *w++ = p;
    }
  }
  return MB_OK;
}

mb_status mb_sched_load(const int64_t *buf, int64_t len, mb_sched **out) {
  if (!buf || !out || len < kStateHeaderWords) return mb::fail(MB_EINVAL, "mb_sched_load: null or short state");
  if (buf[0] != kStateMagic || buf[1] != kStateVersion)
    return mb::fail(MB_EINVAL, "mb_sched_load: not a packer state of this version");
  int64_t at = 2;
  auto word = [&](int64_t lo, int64_t hi, int64_t *v) {
    if (at >= len) return false;
    *v = buf[at++];
    return *v >= lo && *v <= hi;
  };
  int64_t budget, max_seqs, chunk_cap, num_pages, ad[4], n_free;
  if (!word(1, INT32_MAX, &budget) || !word(1, INT32_MAX, &max_seqs) || !word(0, INT32_MAX, &chunk_cap) ||
      !word(0, INT32_MAX, &num_pages) || !word(0, INT32_MAX, &ad[0]) || !word(0, INT32_MAX, &ad[1]) ||
      !word(0, INT32_MAX, &ad[2]) || !word(0, INT32_MAX, &ad[3]) || !word(0, num_pages, &n_free))
    return mb::fail(MB_EINVAL, "mb_sched_load: bad configuration words");
  // every page appears once (free or in a table), so the words bound num_pages
  if (num_pages > len - kStateHeaderWords - 3) return mb::fail(MB_EINVAL, "mb_sched_load: truncated state");
  const bool ad_off = ad[0] == 0 && ad[1] == 0 && ad[2] == 0 && ad[3] == 0;
  if (!ad_off && !(ad[0] >= 1 && ad[1] >= ad[0] && ad[2] >= ad[1] && ad[3] >= 1))
    return mb::fail(MB_EINVAL, "mb_sched_load: bad adaptive chunk settings");
  std::vector<char> seen(static_cast<size_t>(num_pages), 0);
  auto page = [&](int32_t *p) {
    int64_t v;
    if (!word(0, num_pages - 1, &v) || seen[static_cast<size_t>(v)]) return false;
    seen[static_cast<size_t>(v)] = 1;
    *p = static_cast<int32_t>(v);
    return true;
  };
  mb_sched *s = new (std::nothrow) mb_sched();
  if (!s) return mb::fail(MB_ENOMEM, "mb_sched_load: out of host memory");
  s->cfg = {static_cast<int32_t>(budget), static_cast<int32_t>(max_seqs), static_cast<int32_t>(chunk_cap)};
  s->num_pages = static_cast<int32_t>(num_pages);
  s->ad_min = static_cast<int32_t>(ad[0]);
  s->ad_base = static_cast<int32_t>(ad[1]);
  s->ad_max = static_cast<int32_t>(ad[2]);
  s->ad_pressure = static_cast<int32_t>(ad[3]);
  auto reject = [&](const char *what) {
    delete s;
    return mb::fail(MB_EINVAL, "mb_sched_load: %s", what);
  };
  for (int64_t i = 0; i < n_free; ++i) {
    int32_t p;
    if (!page(&p)) return reject("free list holds a page twice or out of range");
    s->free_pages.push_back(p);
  }
  std::list<Req *> *queues[3] = {&s->running, &s->partial, &s->waiting};
  for (int state = 2; state >= 0; --state) {   // running, partial, waiting
    int64_t n;
    if (!word(0, INT32_MAX, &n)) return reject("bad queue length");
    for (int64_t i = 0; i < n; ++i) {
      int64_t id, prompt_len, computed, np;
      if (!word(INT64_MIN, INT64_MAX, &id) || !word(1, INT32_MAX, &prompt_len) ||
          !word(0, INT32_MAX, &computed) || !word(0, num_pages, &np))
        return reject("bad request words");
      const bool fits = state == 0 ? computed == 0 : state == 1 ? computed > 0 && computed < prompt_len
                                                                 : computed >= prompt_len;
      if (!fits) return reject("a request's progress does not match its queue");
      // in 64 bits: the page count of a large `computed` must not wrap
      if (np != (computed + kPage - 1) / kPage) return reject("a request does not hold ceil(computed / 16) pages");
      if (s->by_id.count(id)) return reject("duplicate request id");
      Req *r = new (std::nothrow) Req{id, static_cast<int32_t>(prompt_len), computed, {}, state};
      if (!r) return reject("out of host memory");
      s->by_id[id] = r;
      queues[2 - state]->push_back(r);
      for (int64_t k = 0; k < np; ++k) {
        int32_t p;
        if (!page(&p)) return reject("a block table holds a page twice or out of range");
        r->pages.push_back(p);
      }
    }
  }
  if (at != len) return reject("trailing words after the state");
  for (char c : seen)
    if (!c) return reject("a page is neither free nor held by a request");
  *out = s;
  return MB_OK;
}

mb_status mb_sched_destroy(mb_sched *s) {
  delete s;
  return MB_OK;
}

}  // extern "C"
