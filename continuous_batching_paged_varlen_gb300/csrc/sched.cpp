// Host iteration builder (include/mb_sched.h): which requests run this
// iteration, how many Q rows each, which KV pages they write and read.
//
// Iteration-level scheduling with chunked prefill under a Q-row budget
// ("ORCA and chunked prefill", sections 2-5), decode steps of one row (or
// k + 1) that reuse their tail page, preemption of the latest admitted request
// when the KV pool runs short, and prefix pages shared by reference count
// ("GLM-5.3 e2e token ledger", stage 3; "How To Scale Your Model notes (7-8)",
// section 3). Host memory only.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <new>
#include <vector>

#include "../../include/mb.h"
#include "../../include/mb_sched.h"

namespace {

struct Req {
  int32_t id = 0, prompt_len = 0, max_new = 0, prefix_id = -1, prefix_len = 0;
  int32_t state = MB_SCHED_WAITING;
  int32_t computed = 0;   // positions whose K/V are in the cache
  int32_t generated = 0;  // output tokens so far
  int32_t preemptions = 0;
  int64_t admit_seq = -1;
  std::vector<int32_t> pages;  // block table; prefix pages are shared references
};

struct PrefixEntry {
  std::vector<int32_t> pages;
  int32_t len = 0;  // positions the pages hold (a request hits only on this exact length)
  int64_t last_use = 0;
};

struct Scheduled {
  int32_t id, rows;
};

}  // namespace

struct mb_sched {
  mb_sched_config_t cfg;
  std::vector<Req> reqs;
  std::vector<int32_t> waiting;  // ids, ascending (arrival order)
  std::vector<int32_t> running;  // ids, admission order
  std::vector<int32_t> refs;     // per page
  std::vector<int32_t> free_list;
  std::map<int32_t, PrefixEntry> prefixes;
  std::vector<Scheduled> step;
  bool pending = false;
  int64_t seq = 0;
  int32_t n_finished = 0;
};

namespace {

bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

void release(mb_sched* s, int32_t page) {
  if (--s->refs[page] == 0) s->free_list.push_back(page);
}

// pages a prefix entry could give back (held by the entry alone)
int32_t evictable(const mb_sched* s) {
  int32_t n = 0;
  for (const auto& kv : s->prefixes) {
    bool alone = true;
    for (int32_t p : kv.second.pages) alone = alone && s->refs[p] == 1;
    if (alone) n += (int32_t)kv.second.pages.size();
  }
  return n;
}

// drop the least recently used prefix entry that no request holds
bool evict_one(mb_sched* s) {
  auto best = s->prefixes.end();
  for (auto it = s->prefixes.begin(); it != s->prefixes.end(); ++it) {
    bool alone = true;
    for (int32_t p : it->second.pages) alone = alone && s->refs[p] == 1;
    if (alone && (best == s->prefixes.end() || it->second.last_use < best->second.last_use))
      best = it;
  }
  if (best == s->prefixes.end()) return false;
  for (int32_t p : best->second.pages) release(s, p);
  s->prefixes.erase(best);
  return true;
}

int32_t available(const mb_sched* s) { return (int32_t)s->free_list.size() + evictable(s); }

// allocate pages so that r holds the blocks of positions [0, upto); all or none
bool grow(mb_sched* s, Req& r, int32_t upto) {
  const int32_t need = (upto + s->cfg.page_size - 1) / s->cfg.page_size - (int32_t)r.pages.size();
  if (need <= 0) return true;
  if (need > available(s)) return false;
  for (int32_t k = 0; k < need; ++k) {
    if (s->free_list.empty() && !evict_one(s)) return false;  // cannot happen after the check
    const int32_t p = s->free_list.back();
    s->free_list.pop_back();
    s->refs[p] = 1;
    r.pages.push_back(p);
  }
  return true;
}

// positions r could still cover with its pages and the free / evictable ones
int32_t room(const mb_sched* s, const Req& r) {
  return ((int32_t)r.pages.size() + available(s)) * s->cfg.page_size - r.computed;
}

void drop_pages(mb_sched* s, Req& r) {
  for (int32_t p : r.pages) release(s, p);
  r.pages.clear();
}

void insert_waiting(mb_sched* s, int32_t id) {
  s->waiting.insert(std::lower_bound(s->waiting.begin(), s->waiting.end(), id), id);
}

void preempt(mb_sched* s, int32_t id) {
  Req& r = s->reqs[id];
  drop_pages(s, r);
  r.state = MB_SCHED_WAITING;
  r.computed = 0;
  r.generated = 0;
  r.admit_seq = -1;
  ++r.preemptions;
  s->running.erase(std::find(s->running.begin(), s->running.end(), id));
  insert_waiting(s, id);
}

bool scheduled(const mb_sched* s, int32_t id) {
  for (const Scheduled& e : s->step)
    if (e.id == id) return true;
  return false;
}

}  // namespace

extern "C" {

mb_status_t mb_sched_create(const mb_sched_config_t* cfg, mb_sched_t** out) {
  if (!cfg || !out) return MB_ERR_INVALID_ARG;
  if (cfg->num_pages <= 0 || cfg->max_blocks_per_req <= 0 || cfg->token_budget <= 0 ||
      cfg->max_running < 0 || cfg->decode_rows < 0 || !pow2_in(cfg->page_size, 16, 128))
    return MB_ERR_INVALID_ARG;
  mb_sched* s = new (std::nothrow) mb_sched();
  if (!s) return MB_ERR_INVALID_ARG;
  s->cfg = *cfg;
  if (s->cfg.decode_rows == 0) s->cfg.decode_rows = 1;
  if (s->cfg.decode_rows > s->cfg.token_budget) {
    delete s;
    return MB_ERR_INVALID_ARG;
  }
  s->refs.assign(cfg->num_pages, 0);
  s->free_list.reserve(cfg->num_pages);
  for (int32_t p = cfg->num_pages - 1; p >= 0; --p) s->free_list.push_back(p);
  *out = s;
  return MB_OK;
}

mb_status_t mb_sched_destroy(mb_sched_t* s) {
  delete s;
  return MB_OK;
}

mb_status_t mb_sched_add(mb_sched_t* s, int32_t prompt_len, int32_t max_new_tokens,
                         int32_t prefix_id, int32_t prefix_len, int32_t* request_id) {
  if (!s || !request_id || prompt_len <= 0 || max_new_tokens <= 0 || prefix_id < -1)
    return MB_ERR_INVALID_ARG;
  if (prefix_id >= 0 &&
      (prefix_len <= 0 || prefix_len % s->cfg.page_size != 0 || prefix_len >= prompt_len))
    return MB_ERR_INVALID_ARG;
  // its whole context: the prompt and every output token but the last
  const int64_t ctx = (int64_t)prompt_len + max_new_tokens - 1 + s->cfg.decode_rows - 1;
  const int64_t blocks = (ctx + s->cfg.page_size - 1) / s->cfg.page_size;
  if (blocks > s->cfg.max_blocks_per_req || blocks > s->cfg.num_pages) return MB_ERR_SHAPE;
  Req r;
  r.id = (int32_t)s->reqs.size();
  r.prompt_len = prompt_len;
  r.max_new = max_new_tokens;
  r.prefix_id = prefix_id;
  r.prefix_len = prefix_id >= 0 ? prefix_len : 0;
  s->reqs.push_back(r);
  s->waiting.push_back(r.id);  // ids grow, so the list stays sorted
  *request_id = r.id;
  return MB_OK;
}

mb_status_t mb_sched_step(mb_sched_t* s, mb_request_t* reqs_out, int32_t* ids_out,
                          int32_t* block_table_out, int32_t* slots_out,
                          int32_t* positions_out, int32_t cap_reqs, int32_t cap_rows,
                          mb_sched_stats_t* stats) {
  if (!s || s->pending) return MB_ERR_INVALID_ARG;
  if (cap_reqs < 0 || cap_rows < 0) return MB_ERR_INVALID_ARG;
  const int32_t live = (int32_t)(s->running.size() + s->waiting.size());
  if (cap_reqs < live || cap_rows < std::min<int32_t>(s->cfg.token_budget, 1 << 30))
    return MB_ERR_WORKSPACE;
  if ((live > 0 && (!reqs_out || !ids_out || !block_table_out)) ||
      (cap_rows > 0 && (!slots_out || !positions_out)))
    return MB_ERR_INVALID_ARG;

  const mb_sched_config_t& c = s->cfg;
  s->step.clear();
  int32_t budget = c.token_budget;
  int32_t n_preempted = 0, n_prefix_hits = 0, n_decode = 0, n_prefill = 0;

  // 1. decode steps, admission order; the latest admitted request not yet
  //    scheduled is preempted while the pool cannot hold the next step
  const std::vector<int32_t> order = s->running;
  for (int32_t id : order) {
    Req& r = s->reqs[id];
    if (r.state != MB_SCHED_DECODE) continue;
    if (budget < c.decode_rows) break;
    bool ok = grow(s, r, r.computed + c.decode_rows);
    while (!ok) {
      int32_t victim = -1;
      int64_t latest = -1;
      for (int32_t v : s->running)
        if (!scheduled(s, v) && s->reqs[v].admit_seq > latest) {
          latest = s->reqs[v].admit_seq;
          victim = v;
        }
      if (victim < 0) break;
      preempt(s, victim);
      ++n_preempted;
      if (victim == id) break;
      ok = grow(s, r, r.computed + c.decode_rows);
    }
    if (!ok) continue;  // this request was preempted (or nothing fits)
    s->step.push_back({id, c.decode_rows});
    budget -= c.decode_rows;
    ++n_decode;
  }

  // 2. prefill chunks of admitted requests, admission order
  for (int32_t id : std::vector<int32_t>(s->running)) {
    if (budget <= 0) break;
    Req& r = s->reqs[id];
    if (r.state != MB_SCHED_PREFILL) continue;
    const int32_t chunk = std::min({r.prompt_len - r.computed, budget, room(s, r)});
    if (chunk <= 0 || !grow(s, r, r.computed + chunk)) continue;
    s->step.push_back({id, chunk});
    budget -= chunk;
    ++n_prefill;
  }

  // 3. admissions, first come first served (none in a step that had to
  //    preempt: the pool is short, and the victim would be readmitted at once)
  while (n_preempted == 0 && !s->waiting.empty() && budget > 0 &&
         (c.max_running == 0 || (int32_t)s->running.size() < c.max_running)) {
    const int32_t id = s->waiting.front();
    Req& r = s->reqs[id];
    bool hit = false;
    if (r.prefix_id >= 0) {
      auto it = s->prefixes.find(r.prefix_id);
      if (it != s->prefixes.end() && it->second.len == r.prefix_len) {
        for (int32_t p : it->second.pages) {
          ++s->refs[p];
          r.pages.push_back(p);
        }
        it->second.last_use = s->seq;
        r.computed = r.prefix_len;
        hit = true;
      }
    }
    const int32_t chunk = std::min({r.prompt_len - r.computed, budget, room(s, r)});
    if (chunk <= 0 || !grow(s, r, r.computed + chunk)) {
      drop_pages(s, r);  // undo the prefix references; it waits its turn
      r.computed = 0;
      break;
    }
    s->waiting.erase(s->waiting.begin());
    r.state = MB_SCHED_PREFILL;
    r.admit_seq = s->seq++;
    s->running.push_back(id);
    s->step.push_back({id, chunk});
    budget -= chunk;
    ++n_prefill;
    n_prefix_hits += hit;
  }

  // outputs: flat Q layout in scheduling order
  int32_t q = 0;
  const int32_t ps = c.page_size, mb = c.max_blocks_per_req;
  for (size_t k = 0; k < s->step.size(); ++k) {
    const Req& r = s->reqs[s->step[k].id];
    const int32_t rows = s->step[k].rows;
    reqs_out[k].q_start = q;
    reqs_out[k].q_end = q + rows;
    reqs_out[k].kv_length = r.computed + rows;
    ids_out[k] = r.id;
    int32_t* bt = block_table_out + k * (size_t)mb;
    for (int32_t b = 0; b < mb; ++b) bt[b] = b < (int32_t)r.pages.size() ? r.pages[b] : -1;
    for (int32_t j = 0; j < rows; ++j) {
      const int32_t pos = r.computed + j;
      positions_out[q + j] = pos;
      slots_out[q + j] = r.pages[pos / ps] * ps + pos % ps;
    }
    q += rows;
  }
  s->pending = true;
  if (stats) {
    stats->n_reqs = (int32_t)s->step.size();
    stats->total_q = q;
    stats->n_prefill = n_prefill;
    stats->n_decode = n_decode;
    stats->n_preempted = n_preempted;
    stats->n_prefix_hits = n_prefix_hits;
    stats->n_waiting = (int32_t)s->waiting.size();
    stats->n_running = (int32_t)s->running.size();
    stats->n_finished = s->n_finished;
    stats->free_pages = (int32_t)s->free_list.size();
  }
  return MB_OK;
}

mb_status_t mb_sched_commit(mb_sched_t* s, int32_t* finished_out, int32_t cap,
                            int32_t* n_finished) {
  if (!s || !s->pending || cap < 0) return MB_ERR_INVALID_ARG;
  int32_t nf = 0;
  for (const Scheduled& e : s->step) {
    Req& r = s->reqs[e.id];
    r.computed += e.rows;
    if (r.state == MB_SCHED_PREFILL) {
      if (r.prefix_id >= 0 && r.computed >= r.prefix_len &&
          s->prefixes.find(r.prefix_id) == s->prefixes.end()) {
        // the prefix is in the cache now: keep its pages for later requests
        PrefixEntry pe;
        pe.len = r.prefix_len;
        pe.last_use = s->seq;
        for (int32_t b = 0; b < r.prefix_len / s->cfg.page_size; ++b) {
          ++s->refs[r.pages[b]];
          pe.pages.push_back(r.pages[b]);
        }
        s->prefixes[r.prefix_id] = pe;
      }
      if (r.computed == r.prompt_len) {
        r.state = MB_SCHED_DECODE;
        r.generated = 1;  // the last prompt position's logits give the first token
      }
    } else if (r.state == MB_SCHED_DECODE) {
      r.generated += e.rows;
    }
    if (r.state == MB_SCHED_DECODE && r.generated >= r.max_new) {
      drop_pages(s, r);
      r.state = MB_SCHED_FINISHED;
      s->running.erase(std::find(s->running.begin(), s->running.end(), r.id));
      ++s->n_finished;
      if (finished_out && nf < cap) finished_out[nf] = r.id;
      ++nf;
    }
  }
  s->step.clear();
  s->pending = false;
  if (n_finished) *n_finished = nf;
  return MB_OK;
}

mb_status_t mb_sched_page_refs(const mb_sched_t* s, int32_t* refs_out, int32_t num_pages) {
  if (!s || !refs_out || num_pages != s->cfg.num_pages) return MB_ERR_INVALID_ARG;
  memcpy(refs_out, s->refs.data(), sizeof(int32_t) * (size_t)num_pages);
  return MB_OK;
}

mb_status_t mb_sched_request_info(const mb_sched_t* s, int32_t request_id, int32_t* info_out) {
  if (!s || !info_out || request_id < 0 || request_id >= (int32_t)s->reqs.size())
    return MB_ERR_INVALID_ARG;
  const Req& r = s->reqs[request_id];
  info_out[0] = r.state;
  info_out[1] = r.computed;
  info_out[2] = r.generated;
  info_out[3] = (int32_t)r.pages.size();
  info_out[4] = r.preemptions;
  info_out[5] = r.prompt_len;
  info_out[6] = r.max_new;
  info_out[7] = r.prefix_id;
  return MB_OK;
}

}  // extern "C"
