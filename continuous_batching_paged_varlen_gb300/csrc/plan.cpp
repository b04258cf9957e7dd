// Host planner: validation, request classification, shared-prefix grouping,
// split-KV chunking and workspace layout for one iteration.
//
// The triple (q_start, q_end, kv_length) and the two-block mask follow
// "ORCA and chunked prefill", sections 2 and 4; pages shared between
// requests and the "load a common block once for every request that uses
// it" cascade follow "How To Scale Your Model notes (7-8)", section 3.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/mb.h"
#include "mb_internal.h"
#include "plan_impl.h"

using namespace mb;

namespace {

constexpr int kDefaultPrefillMinRows = 16;
// SMs of the GPU the planner sizes work for (a GB300); the split-KV kernel
// keeps one CTA per SM
constexpr int kSms = 152;
// split-KV CTAs to aim for on large batches (~2 waves)
constexpr int kDefaultTargetCtas = 2 * kSms;
// shortest automatic split-KV chunk on large batches: 8 key tiles amortise a
// CTA's set-up
constexpr int kMinChunk = 1024;
// A batch with at most this many 128-key tiles of split-KV work (summed over
// CTAs as if unsplit) is latency-bound: its chunks are sized so that the CTAs
// fill one wave of SMs with as few tiles each as possible (but at least
// kMinSmallChunk keys, so set-up stays a minority of a CTA's time).
constexpr int64_t kSmallBatchTiles = (int64_t)kSms * 8;
constexpr int kMinSmallChunk = 256;

// Cost model of a mixed iteration (both kernels), measured on a GB300 at the
// maximum SM clock: one 128-key tile of one 128-row query tile on the
// tensor-core prefill kernel (D = 128; the issue-bound kernel runs D / 16 + 8
// MMAs per tile), a prefill work item's fixed cost, the rate at which one SM
// of the split-KV kernel streams K/V when HBM is not the limit, and the HBM
// rate the split-KV kernel reaches on the whole GPU.
constexpr double kPrefillTileUs = 0.85;
constexpr double kPrefillItemUs = 2.0;
constexpr double kDecodeSmGBs = 60.0;
constexpr double kHbmGBs = 6600.0;
// the same two rates for the split-KV kernel over an fp8 cache
constexpr double kDecodeFp8SmGBs = 26.0;
constexpr double kHbmFp8GBs = 3950.0;
// A small split-KV batch beside prefill work is latency-bound: each CTA takes
// a fixed time (set-up, its first tiles' latency, epilogue) plus a time per
// 128-key tile that its ring, not HBM, sets; beside it, a prefill item costs
// more than the tile model above counts (the item's Q load, ramp and
// epilogue). Fitted to measured steps of the Llama-2-7B-shaped iteration
// over prefill grids of 120-152 CTAs and two chunkings (rms 4.5 us); the fp8
// split-KV kernel's short CTAs measured the same (same best grid and chunk).
constexpr double kDecodeCtaUs = 14.0;
constexpr double kDecodeTileUs = 1.7;
constexpr double kPrefillItemLatencyUs = 9.0;

bool is_pow2_in(int v, int lo, int hi) {
  return v >= lo && v <= hi && (v & (v - 1)) == 0;
}

}  // namespace

namespace mb {

mb_status_t validate_config(const mb_config_t* cfg) {
  if (!cfg) return MB_ERR_INVALID_ARG;
  if (cfg->n_q_heads <= 0 || cfg->n_kv_heads <= 0 || cfg->num_pages <= 0 ||
      cfg->max_blocks_per_req <= 0 || cfg->page_size <= 0 || cfg->head_dim <= 0)
    return MB_ERR_SHAPE;
  if (cfg->n_q_heads % cfg->n_kv_heads != 0) return MB_ERR_SHAPE;
  if (!(cfg->scale >= 0.0f) || !isfinite(cfg->scale)) return MB_ERR_INVALID_ARG;
  if (cfg->head_dim != 64 && cfg->head_dim != 128) return MB_ERR_UNSUPPORTED;
  if (!is_pow2_in(cfg->page_size, 16, 128)) return MB_ERR_UNSUPPORTED;
  // element offsets of the caches must fit the kernels' 64-bit math and the
  // tensor-map row coordinate (int32)
  int64_t rows = (int64_t)cfg->num_pages * cfg->n_kv_heads * cfg->page_size;
  if (rows >= ((int64_t)1 << 31)) return MB_ERR_UNSUPPORTED;
  return MB_OK;
}

mb_status_t validate_requests(const mb_request_t* reqs, int32_t n,
                              const int32_t* bt, const mb_config_t* cfg,
                              int32_t* total_q_out) {
  if (n < 0) return MB_ERR_INVALID_ARG;
  if (n > 0 && (!reqs || !bt)) return MB_ERR_INVALID_ARG;
  const int ps = cfg->page_size;
  int32_t total_q = 0;
  std::vector<std::pair<int32_t, int32_t>> ranges;
  for (int32_t r = 0; r < n; ++r) {
    const mb_request_t& q = reqs[r];
    if (q.q_start < 0 || q.q_end < q.q_start || q.kv_length < 0) return MB_ERR_SHAPE;
    const int32_t m = q.q_end - q.q_start;
    if (m > q.kv_length) return MB_ERR_SHAPE;
    if (m == 0) continue;
    const int64_t blocks = ((int64_t)q.kv_length + ps - 1) / ps;
    if (blocks > cfg->max_blocks_per_req) return MB_ERR_SHAPE;
    const int32_t* row = bt + (size_t)r * cfg->max_blocks_per_req;
    for (int64_t b = 0; b < blocks; ++b)
      if (row[b] < 0 || row[b] >= cfg->num_pages) return MB_ERR_SHAPE;
    ranges.push_back({q.q_start, q.q_end});
    total_q = std::max(total_q, q.q_end);
  }
  std::sort(ranges.begin(), ranges.end());
  for (size_t i = 1; i < ranges.size(); ++i)
    if (ranges[i].first < ranges[i - 1].second) return MB_ERR_SHAPE;
  if ((int64_t)total_q * cfg->n_q_heads * cfg->head_dim >= ((int64_t)1 << 40))
    return MB_ERR_UNSUPPORTED;
  *total_q_out = total_q;
  return MB_OK;
}

namespace {

struct Sequence {       // one key range walked by split-KV CTAs
  int32_t bt_row;
  int32_t k_begin, k_end;
  int32_t mbeg, mend;   // requests whose rows attend to it: member_list[mbeg, mend)
  bool shared;
};

// Indices 0..n-1 ordered by key (>= 0) descending, ties in index order (the
// plan's heaviest-first CTA order): a stable counting sort over the key range
// when it is small (keys are tile or key counts), else one sort of packed
// 64-bit keys; the work items themselves are moved once, by the caller.
template <typename KeyFn>
std::vector<int32_t> heavy_first(size_t n, KeyFn key) {
  std::vector<int32_t> order(n);
  int32_t kmax = 0;
  for (size_t i = 0; i < n; ++i) kmax = std::max(kmax, key(i));
  if (kmax <= (int32_t)std::max<size_t>(4 * n, 1 << 16)) {
    std::vector<int32_t> start((size_t)kmax + 2, 0);
    for (size_t i = 0; i < n; ++i) ++start[(size_t)(kmax - key(i)) + 1];
    for (size_t b = 1; b < start.size(); ++b) start[b] += start[b - 1];
    for (size_t i = 0; i < n; ++i) order[start[(size_t)(kmax - key(i))]++] = (int32_t)i;
    return order;
  }
  std::vector<uint64_t> k(n);
  for (size_t i = 0; i < n; ++i)
    k[i] = ((uint64_t)(uint32_t)(INT32_MAX - key(i)) << 32) | (uint32_t)i;
  std::sort(k.begin(), k.end());
  for (size_t i = 0; i < n; ++i) order[i] = (int32_t)(k[i] & 0xffffffffu);
  return order;
}

// Modelled cost of each prefill item (us): a fixed cost per item plus its
// query tiles' KV tiles (one 128-row query tile against one 128-key tile).
std::vector<double> prefill_costs(const std::vector<PrefillItem>& pitems, int D, double item_us) {
  const double tile_us = kPrefillTileUs * (D / 16 + 8) / 16.0;
  std::vector<double> cost(pitems.size());
  for (size_t i = 0; i < pitems.size(); ++i) {
    const PrefillItem& p = pitems[i];
    const int32_t ra = std::min(kPrefillTileM, p.n_rows), rb = std::max(0, p.n_rows - kPrefillTileM);
    const int32_t na = (std::min(p.kv_length, p.s0 + p.i0 + ra) + kPrefillTileN - 1) / kPrefillTileN;
    const int32_t nb = rb > 0 ? (std::min(p.kv_length, p.s0 + p.i0 + kPrefillTileM + rb) +
                                 kPrefillTileN - 1) / kPrefillTileN
                              : 0;
    cost[i] = item_us + (na + nb) * tile_us;
  }
  return cost;
}

// Finishing time of each of P prefill CTAs: the items, heavy first, dealt
// in the kernel's snake order (ascending when `sorted`).
void prefill_finish(const std::vector<double>& cost, int32_t P, std::vector<double>& load,
                    bool sorted = true) {
  const int32_t n = (int32_t)cost.size();
  load.assign((size_t)P, 0.0);
  for (int32_t k = 0; k * P < n; ++k)
    for (int32_t b = 0; b < P; ++b) {
      const int32_t idx = k * P + ((k & 1) ? P - 1 - b : b);
      if (idx < n) load[(size_t)b] += cost[(size_t)idx];
    }
  if (sorted) std::sort(load.begin(), load.end());
}

// SMs for the persistent prefill grid when the split-KV kernel runs beside
// it: the grid P whose modelled step time is least (the largest such P on a
// tie). The prefill items (heavy first) go to P CTAs in snake order, which
// gives each CTA its finishing time. Over time the split-KV kernel has the
// kSms - P SMs without a prefill CTA, plus every prefill SM whose CTA has
// finished (its CTAs are handed out as SMs free up); it streams at sm_gbs
// per SM, never faster than full_gbs. The step ends when both are done.
int32_t partition_sms(const std::vector<PrefillItem>& pitems, int64_t decode_bytes, int D,
                      double sm_gbs, double full_gbs) {
  const int32_t n = (int32_t)pitems.size();
  const int32_t hi = std::min<int32_t>(n, kSms), lo = std::max<int32_t>(1, hi / 4);
  const std::vector<double> cost = prefill_costs(pitems, D, kPrefillItemUs);
  const double bytes_per_us_sm = sm_gbs * 1e3, bytes_per_us_full = full_gbs * 1e3;
  std::vector<double> load;
  auto step_of = [&](int32_t P) {
    prefill_finish(cost, P, load);
    const double t_pre = load.back();
    // walk the intervals between prefill CTAs' finishing times
    double left = (double)decode_bytes, t = 0.0, t_dec = -1.0;
    int32_t free_sms = kSms - P;
    for (int32_t b = 0; b <= P && t_dec < 0.0; ++b) {
      const double t_next = b < P ? load[(size_t)b] : 1e300;
      const double rate = std::min(bytes_per_us_full, free_sms * bytes_per_us_sm);
      if (rate > 0.0 && left <= rate * (t_next - t)) t_dec = t + left / rate;
      else if (rate > 0.0) left -= rate * (t_next - t);
      t = t_next;
      ++free_sms;
    }
    return std::max(t_pre, t_dec);
  };
  // every 4th grid size from the full one down, then every size around the
  // best of those (the modelled time is nearly smooth in P)
  int32_t best = hi;
  double best_t = 1e300;
  auto consider = [&](int32_t P) {
    const double st = step_of(P);
    if (st < best_t * (1.0 - 1e-3) || (st < best_t * (1.0 + 1e-3) && P > best)) {
      if (st < best_t) best_t = st;
      best = P;
    }
  };
  for (int32_t P = hi; P >= lo; P -= 4) consider(P);
  const int32_t c = best;
  for (int32_t P = std::min(hi, c + 3); P >= std::max(lo, c - 3); --P)
    if (P != c && (c - P) % 4 != 0) consider(P);
  return best;
}

// The same choice for a small (latency-bound) split-KV batch, whose CTAs
// (tiles[i] 128-key tiles each, heaviest first, the order the hardware hands
// them out) take kDecodeCtaUs + tiles * kDecodeTileUs each: they go, in
// order, to the earliest free SM among the kSms - P without a prefill CTA and
// the prefill SMs as their CTAs finish. The list schedule only changes where
// ceil(CTAs / free SMs) does, so P is tried there and at the full grid.
// Returns the modelled step time (us) and the best P in *best_p.
double latency_partition(const std::vector<double>& cost, const std::vector<int32_t>& tiles,
                         int32_t* best_p) {
  const int32_t n = (int32_t)cost.size();
  const int32_t hi = std::min<int32_t>(n, kSms), lo = std::max<int32_t>(1, hi / 4);
  const int32_t C = (int32_t)tiles.size();
  double total = 0.0;
  for (double c : cost) total += c;
  const double cta_max = kDecodeCtaUs + (C ? tiles[0] : 0) * kDecodeTileUs;
  // candidates: the full grid, and of the grids where the CTAs' wave count
  // on the free SMs changes, the three whose rough estimate (balanced
  // prefill, whole waves of the longest CTA) is least
  std::vector<std::pair<double, int32_t>> est;
  for (int32_t wv = 1; wv <= std::min<int32_t>(C, 64); ++wv) {
    const int32_t P = kSms - (C + wv - 1) / wv;
    if (P < lo || P >= hi) continue;
    const double e = std::max(total / P, wv * cta_max);
    if (est.empty() || est.back().second != P) est.emplace_back(e, P);
  }
  std::sort(est.begin(), est.end());
  std::vector<int32_t> cand{hi};
  for (size_t i = 0; i < est.size() && i < 3; ++i) cand.push_back(est[i].second);
  std::sort(cand.begin(), cand.end(), std::greater<int32_t>());
  double best_t = 1e300;
  *best_p = hi;
  std::vector<double> load;
  for (int32_t P : cand) {
    prefill_finish(cost, P, load, false);
    const double t_pre = *std::max_element(load.begin(), load.end());
    load.insert(load.end(), (size_t)(kSms - P), 0.0);
    std::make_heap(load.begin(), load.end(), std::greater<double>());
    double t_dec = 0.0;
    for (int32_t t : tiles) {
      std::pop_heap(load.begin(), load.end(), std::greater<double>());
      const double e = load.back() + kDecodeCtaUs + t * kDecodeTileUs;
      load.back() = e;
      std::push_heap(load.begin(), load.end(), std::greater<double>());
      t_dec = std::max(t_dec, e);
    }
    const double step = std::max(t_pre, t_dec);
    if (step < best_t * (1.0 - 1e-3)) {
      best_t = step;
      *best_p = P;
    }
  }
  return best_t;
}

}  // namespace

mb_status_t build_plan(const mb_request_t* reqs, int32_t n,
                       const int32_t* bt, const mb_config_t* cfg,
                       const mb_plan_options_t* opts, mb_plan* plan) {
  mb_status_t st = validate_config(cfg);
  if (st != MB_OK) return st;
  int32_t total_q = 0;
  st = validate_requests(reqs, n, bt, cfg, &total_q);
  if (st != MB_OK) return st;

  mb_plan_options_t o = {};
  if (opts) o = *opts;
  if (o.kv_chunk < 0 || (o.kv_chunk % 64) != 0 || o.target_ctas < 0)
    return MB_ERR_INVALID_ARG;
  if (o.prefill_ctas > kSms) o.prefill_ctas = kSms;
  const int prefill_min = o.prefill_min_rows == 0 ? kDefaultPrefillMinRows
                                                  : o.prefill_min_rows;
  const int target = o.target_ctas ? o.target_ctas : kDefaultTargetCtas;

  const int Hq = cfg->n_q_heads, Hkv = cfg->n_kv_heads, g = Hq / Hkv;
  const int ps = cfg->page_size, D = cfg->head_dim;
  const int mb = cfg->max_blocks_per_req;

  std::vector<int32_t> prefill_reqs, decode_reqs;
  for (int32_t r = 0; r < n; ++r) {
    const int32_t m = reqs[r].q_end - reqs[r].q_start;
    if (m == 0) continue;
    if (prefill_min > 0 && m >= prefill_min)
      prefill_reqs.push_back(r);
    else
      decode_reqs.push_back(r);
  }

  // ---- shared-prefix groups among split-KV requests -------------------
  // requests are grouped by the physical page of their first block (a sort
  // of (page, request) pairs); a group of two or more then shares the
  // longest run of leading blocks that every member maps to the same pages
  std::vector<int32_t> own_begin(n, 0);
  std::vector<Sequence> seqs;
  std::vector<int32_t> member_list;
  seqs.reserve(decode_reqs.size() + 1);
  member_list.reserve(2 * decode_reqs.size());
  int32_t n_groups = 0, cascade_keys = 0;
  if (!o.disable_cascade) {
    std::vector<uint64_t> firsts;
    firsts.reserve(decode_reqs.size());
    for (int32_t r : decode_reqs) {
      const int32_t s0 = reqs[r].kv_length - (reqs[r].q_end - reqs[r].q_start);
      if (s0 >= ps) firsts.push_back(((uint64_t)(uint32_t)bt[(size_t)r * mb] << 32) | (uint32_t)r);
    }
    std::sort(firsts.begin(), firsts.end());
    for (size_t a = 0; a < firsts.size();) {
      size_t b = a + 1;
      while (b < firsts.size() && (firsts[b] >> 32) == (firsts[a] >> 32)) ++b;
      if (b - a >= 2) {
        const int32_t mbeg = (int32_t)member_list.size();
        for (size_t x = a; x < b; ++x) member_list.push_back((int32_t)(firsts[x] & 0xffffffffu));
        const int32_t mend = (int32_t)member_list.size();
        // longest run of leading blocks that every member maps to the same
        // physical page and that lies wholly inside every member's cache
        int32_t L = 0;
        for (;; ++L) {
          bool ok = true;
          // (L + 1) * ps <= s0 <= kv_length keeps L inside every member's
          // validated block-table entries; check it before reading entry L
          for (int32_t x = mbeg; x < mend && ok; ++x) {
            const int32_t r = member_list[x];
            const int32_t s0 = reqs[r].kv_length - (reqs[r].q_end - reqs[r].q_start);
            if ((int64_t)(L + 1) * ps > s0) ok = false;
          }
          if (!ok) break;
          const int32_t page = bt[(size_t)member_list[mbeg] * mb + L];
          for (int32_t x = mbeg; x < mend && ok; ++x)
            if (bt[(size_t)member_list[x] * mb + L] != page) ok = false;
          if (!ok) break;
        }
        if (L >= 1) {
          Sequence sq;
          sq.bt_row = member_list[mbeg];
          sq.k_begin = 0;
          sq.k_end = L * ps;
          sq.mbeg = mbeg;
          sq.mend = mend;
          sq.shared = true;
          seqs.push_back(sq);
          for (int32_t x = mbeg; x < mend; ++x) own_begin[member_list[x]] = L * ps;
          ++n_groups;
          cascade_keys += L * ps;
        } else {
          member_list.resize(mbeg);
        }
      }
      a = b;
    }
  }
  for (int32_t r : decode_reqs) {
    Sequence sq;
    sq.bt_row = r;
    sq.k_begin = own_begin[r];
    sq.k_end = reqs[r].kv_length;
    sq.mbeg = (int32_t)member_list.size();
    member_list.push_back(r);
    sq.mend = sq.mbeg + 1;
    sq.shared = false;
    seqs.push_back(sq);
  }

  // ---- prefill items, heaviest first -----------------------------------
  std::vector<PrefillItem> pitems;
  {
    size_t np = 0;
    for (int32_t r : prefill_reqs)
      np += (size_t)Hq * ((reqs[r].q_end - reqs[r].q_start + kPrefillCtaRows - 1) / kPrefillCtaRows);
    pitems.reserve(np);
  }
  for (int32_t r : prefill_reqs) {
    const mb_request_t& q = reqs[r];
    const int32_t m = q.q_end - q.q_start, s0 = q.kv_length - m;
    for (int32_t h = 0; h < Hq; ++h)
      for (int32_t i0 = 0; i0 < m; i0 += kPrefillCtaRows) {
        PrefillItem p;
        p.req = r;
        p.q_head = h;
        p.q_row0 = q.q_start + i0;
        p.n_rows = std::min(kPrefillCtaRows, m - i0);
        p.s0 = s0;
        p.i0 = i0;
        p.kv_length = q.kv_length;
        const int32_t last = std::min(q.kv_length, s0 + i0 + p.n_rows);
        p.n_kv_tiles = (last + kPrefillTileN - 1) / kPrefillTileN;
        pitems.push_back(p);
      }
  }
  {
    const std::vector<int32_t> order =
        heavy_first(pitems.size(), [&](size_t i) { return pitems[i].n_kv_tiles; });
    std::vector<PrefillItem> sorted(pitems.size());
    for (size_t i = 0; i < order.size(); ++i) sorted[i] = pitems[order[i]];
    pitems.swap(sorted);
  }

  // ---- split-KV chunk size ---------------------------------------------
  int64_t work = 0;   // key-visits summed over CTAs if nothing were split
  int64_t tiles = 0;  // the same in 128-key tiles
  for (const Sequence& s : seqs) {
    int64_t rows = 0;
    for (int32_t x = s.mbeg; x < s.mend; ++x) {
      const int32_t r = member_list[x];
      rows += (int64_t)(reqs[r].q_end - reqs[r].q_start) * g;
    }
    const int64_t groups = (rows + kRowsPerDecodeItem - 1) / kRowsPerDecodeItem;
    work += (int64_t)(s.k_end - s.k_begin) * groups * Hkv;
    tiles += (int64_t)((s.k_end - s.k_begin + 127) / 128) * groups * Hkv;
  }
  int32_t chunk = o.kv_chunk;
  const bool one_wave = chunk == 0 && o.target_ctas == 0 && tiles <= kSmallBatchTiles;
  if (one_wave) {
    // start from ceil(tiles / SMs) tiles per CTA; the search below grows it
    // until page rounding leaves no CTA for a second wave
    const int64_t per = (tiles + kSms - 1) / kSms;
    chunk = (int32_t)std::max<int64_t>(per * 128, kMinSmallChunk);
  } else if (chunk == 0) {
    int64_t c = (work + target - 1) / std::max(1, target);
    chunk = (int32_t)std::min<int64_t>(std::max<int64_t>(c, kMinChunk), 1 << 30);
  }
  chunk = ((chunk + ps - 1) / ps) * ps;  // chunk boundaries stay page-aligned
  // a key range of length len is cut into ceil(len / chunk) nearly equal
  // page-aligned parts (no sliver of a few keys at the end)
  auto part_of = [&](const Sequence& s) -> int32_t {
    const int32_t len = s.k_end - s.k_begin;
    if (len <= 0) return chunk;
    const int32_t parts = (len + chunk - 1) / chunk;
    const int32_t even = (len + parts - 1) / parts;
    return ((even + ps - 1) / ps) * ps;
  };
  if (one_wave) {
    auto ctas = [&]() -> int64_t {
      int64_t c = 0;
      for (const Sequence& s : seqs) {
        const int32_t len = s.k_end - s.k_begin;
        if (len <= 0) continue;
        int64_t rows = 0;
        for (int32_t x = s.mbeg; x < s.mend; ++x) {
          const int32_t r = member_list[x];
          rows += (int64_t)(reqs[r].q_end - reqs[r].q_start) * g;
        }
        const int64_t groups = (rows + kRowsPerDecodeItem - 1) / kRowsPerDecodeItem;
        c += (int64_t)((len + part_of(s) - 1) / part_of(s)) * groups * Hkv;
      }
      return c;
    };
    const int step = std::max(ps, 128);
    for (int guard = 0; guard < 4096 && ctas() > kSms; ++guard) chunk += step;
  }
  // A small batch beside prefill work: its CTAs are latency-bound, and how
  // many SMs the prefill grid leaves them decides how long they take, so the
  // chunk (sized for one wave of SMs, or every key range whole) is chosen
  // together with the prefill grid's size (latency_partition).
  int32_t latency_p = 0;
  if (one_wave && !pitems.empty() && o.prefill_ctas == 0) {
    const std::vector<double> cost = prefill_costs(pitems, D, kPrefillItemLatencyUs);
    auto cta_tiles = [&]() {
      std::vector<int32_t> t;
      for (const Sequence& s : seqs) {
        const int32_t len = s.k_end - s.k_begin;
        if (len <= 0) continue;
        int64_t rs = 0;
        for (int32_t x = s.mbeg; x < s.mend; ++x) {
          const int32_t r = member_list[x];
          rs += (int64_t)(reqs[r].q_end - reqs[r].q_start) * g;
        }
        const int64_t ctas = ((rs + kRowsPerDecodeItem - 1) / kRowsPerDecodeItem) * Hkv;
        const int32_t part = part_of(s), nc = (len + part - 1) / part;
        for (int32_t c = 0; c < nc; ++c) {
          const int32_t lc = std::min(part, len - c * part);
          t.insert(t.end(), (size_t)ctas, (lc + 127) / 128);
        }
      }
      std::sort(t.begin(), t.end(), std::greater<int32_t>());
      return t;
    };
    int32_t p_wave = 0, p_whole = 0;
    const double t_wave = latency_partition(cost, cta_tiles(), &p_wave);
    const int32_t chunk_wave = chunk;
    int32_t longest = 0;
    for (const Sequence& s : seqs) longest = std::max(longest, s.k_end - s.k_begin);
    chunk = std::max(chunk_wave, ((longest + ps - 1) / ps) * ps);
    const double t_whole = latency_partition(cost, cta_tiles(), &p_whole);
    if (t_whole < t_wave * (1.0 - 1e-3)) {
      latency_p = p_whole;
    } else {
      chunk = chunk_wave;
      latency_p = p_wave;
    }
  }
  auto n_chunks = [&](const Sequence& s) -> int32_t {
    const int32_t len = s.k_end - s.k_begin;
    return len <= 0 ? 0 : (len + part_of(s) - 1) / part_of(s);
  };

  // ---- partial slots per output row ------------------------------------
  // every output row of a split-KV request owns n_slots contiguous partial
  // slots: first the chunks of its shared prefix (if any), then its own.
  std::vector<int32_t> shared_chunks(n, 0), own_chunks(n, 0), slot_base(n, -1);
  for (const Sequence& s : seqs)
    for (int32_t x = s.mbeg; x < s.mend; ++x) {
      const int32_t r = member_list[x];
      if (s.shared)
        shared_chunks[r] = n_chunks(s);
      else
        own_chunks[r] = n_chunks(s);
    }
  int32_t n_partials = 0;
  std::vector<CombineEntry> combine;
  for (int32_t r : decode_reqs) {
    const int32_t slots = shared_chunks[r] + own_chunks[r];
    if (slots <= 1) continue;
    slot_base[r] = n_partials;
    const int32_t m = reqs[r].q_end - reqs[r].q_start;
    for (int32_t i = 0; i < m; ++i)
      for (int32_t h = 0; h < Hq; ++h) {
        CombineEntry e;
        e.q_index = reqs[r].q_start + i;
        e.q_head = h;
        e.slot_begin = n_partials;
        e.n_slots = slots;
        combine.push_back(e);
        n_partials += slots;
      }
  }
  auto slot_of = [&](int32_t r, int32_t i, int32_t hq, bool shared, int32_t c) -> int32_t {
    if (slot_base[r] < 0) return -1;
    const int32_t slots = shared_chunks[r] + own_chunks[r];
    const int32_t idx = shared ? c : shared_chunks[r] + c;
    return slot_base[r] + (i * Hq + hq) * slots + idx;
  };

  // ---- split-KV items and row descriptors -----------------------------
  // per (sequence, KV head, key chunk): the rows of every member request x
  // its new rows x the g query heads of the KV head, 128 rows per CTA
  size_t est_items = 0, est_rows = 0;
  for (const Sequence& s : seqs) {
    int64_t rs = 0;
    for (int32_t x = s.mbeg; x < s.mend; ++x) {
      const int32_t r = member_list[x];
      rs += (int64_t)(reqs[r].q_end - reqs[r].q_start) * g;
    }
    const int64_t nc = n_chunks(s);
    est_items += (size_t)(nc * Hkv * ((rs + kRowsPerDecodeItem - 1) / kRowsPerDecodeItem));
    est_rows += (size_t)(nc * Hkv * rs);
  }
  std::vector<DecodeItem> items;
  std::vector<RowDesc> rows;
  items.reserve(est_items);
  rows.reserve(est_rows);
  for (const Sequence& s : seqs) {
    const int32_t nc = n_chunks(s);
    const int32_t part = part_of(s);
    for (int32_t h = 0; h < Hkv; ++h) {
      for (int32_t c = 0; c < nc; ++c) {
        const int32_t kb = s.k_begin + c * part;
        const int32_t ke = std::min(s.k_end, kb + part);
        DecodeItem it = {};
        it.bt_row = s.bt_row;
        it.kv_head = h;
        it.k_begin = kb;
        it.k_end = ke;
        // a shared prefix lies below every sharer's new rows; a request's own
        // range holds its new rows from S0 on
        it.k_new = s.shared ? ke
                            : std::min(ke, std::max(kb, reqs[s.bt_row].kv_length -
                                                            (reqs[s.bt_row].q_end -
                                                             reqs[s.bt_row].q_start)));
        it.row_begin = (int32_t)rows.size();
        for (int32_t x = s.mbeg; x < s.mend; ++x) {
          const int32_t r = member_list[x];
          const mb_request_t& q = reqs[r];
          const int32_t m = q.q_end - q.q_start, s0 = q.kv_length - m;
          for (int32_t i = 0; i < m; ++i)
            for (int32_t jg = 0; jg < g; ++jg) {
              if ((int32_t)rows.size() - it.row_begin == kRowsPerDecodeItem) {
                it.n_rows = kRowsPerDecodeItem;
                items.push_back(it);
                it.row_begin = (int32_t)rows.size();
              }
              RowDesc d;
              d.q_index = q.q_start + i;
              d.q_head = h * g + jg;
              d.vis_end = s0 + i + 1;
              d.dst = slot_of(r, i, d.q_head, s.shared, c);
              rows.push_back(d);
            }
        }
        it.n_rows = (int32_t)rows.size() - it.row_begin;
        if (it.n_rows > 0) items.push_back(it);
      }
    }
  }

  // heaviest split-KV CTAs first (the hardware hands out CTAs in order)
  {
    const std::vector<int32_t> order =
        heavy_first(items.size(), [&](size_t i) { return items[i].k_end - items[i].k_begin; });
    std::vector<DecodeItem> sorted(items.size());
    for (size_t i = 0; i < order.size(); ++i) sorted[i] = items[order[i]];
    items.swap(sorted);
  }

  // ---- split-KV build: row copies when most keys sit in long CTAs of
  // <= 32 rows (see splitkv_kernel) ---------------------------------------
  int32_t decode_copies = 0, decode_max_rows = 0;
  {
    int64_t long_tiles = 0, all_tiles = 0;
    for (const DecodeItem& it : items) {
      decode_max_rows = std::max(decode_max_rows, it.n_rows);
      const int64_t t = (it.k_end - it.k_begin + 127) / 128;
      all_tiles += t;
      if (t >= kCopyMinTiles && it.n_rows <= 32) long_tiles += t;
    }
    decode_copies = 2 * long_tiles >= all_tiles && all_tiles > 0 ? 1 : 0;
  }

  // ---- SMs of the prefill grid beside the split-KV kernel ---------------
  int32_t prefill_ctas = std::min<int32_t>((int32_t)pitems.size(), kSms);
  if (!pitems.empty() && !items.empty()) {
    if (o.prefill_ctas > 0) {
      prefill_ctas = std::min(prefill_ctas, o.prefill_ctas);
    } else if (o.prefill_ctas == 0 && latency_p > 0) {
      prefill_ctas = std::min(prefill_ctas, latency_p);
    } else if (o.prefill_ctas == 0) {
      // K and V bytes the split-KV CTAs read (fp8: codes and row scales)
      const int64_t per_key = o.fp8_cache ? 2 * (D + 4) : 4 * D;
      int64_t dbytes = 0;
      for (const DecodeItem& it : items) dbytes += (int64_t)(it.k_end - it.k_begin) * per_key;
      prefill_ctas = o.fp8_cache
                         ? partition_sms(pitems, dbytes, D, kDecodeFp8SmGBs, kHbmFp8GBs)
                         : partition_sms(pitems, dbytes, D, kDecodeSmGBs, kHbmGBs);
    }
  }

  // ---- fp8 cache: pages of the prefill requests, staged as bf16 ----------
  // the prefill kernel reads them through stage_bt, a copy of the block
  // table whose prefill rows hold staging page ids; a page several prefill
  // requests map is staged once
  std::vector<int32_t> stage_pages;
  std::vector<int32_t> stage_bt;
  if (o.fp8_cache && !pitems.empty()) {
    std::vector<int32_t> stage_of((size_t)cfg->num_pages, -1);
    stage_bt.assign((size_t)n * mb, 0);
    for (int32_t r : prefill_reqs) {
      const int32_t nb = (reqs[r].kv_length + ps - 1) / ps;
      for (int32_t b = 0; b < nb; ++b) {
        const int32_t page = bt[(size_t)r * mb + b];
        if (stage_of[(size_t)page] < 0) {
          stage_of[(size_t)page] = (int32_t)stage_pages.size();
          stage_pages.push_back(page);
        }
        stage_bt[(size_t)r * mb + b] = stage_of[(size_t)page];
      }
    }
  }

  // ---- workspace layout + host image -----------------------------------
  PlanDevice& d = plan->dev;
  d = PlanDevice{};
  d.n_decode_items = (int32_t)items.size();
  d.n_decode_rows = (int32_t)rows.size();
  d.n_prefill_items = (int32_t)pitems.size();
  d.n_combine = (int32_t)combine.size();
  d.n_partials = n_partials;
  d.n_q_heads = Hq;
  d.n_kv_heads = Hkv;
  d.head_dim = D;
  d.page_size = ps;
  d.num_pages = cfg->num_pages;
  d.max_blocks = mb;
  d.total_q = total_q;
  d.prefill_ctas = pitems.empty() ? 0 : prefill_ctas;
  d.decode_copies = decode_copies;
  d.decode_max_rows = decode_max_rows;
  d.scale = cfg->scale > 0.f ? cfg->scale : 1.0f / sqrtf((float)D);
  size_t off = kStatusBytes;
  d.off_decode_items = off;
  off = align256(off + items.size() * sizeof(DecodeItem));
  d.off_rows = off;
  off = align256(off + rows.size() * sizeof(RowDesc));
  d.off_prefill_items = off;
  off = align256(off + pitems.size() * sizeof(PrefillItem));
  d.off_combine = off;
  off = align256(off + combine.size() * sizeof(CombineEntry));
  // per decode row its merge reference, then one arrival counter per entry
  // (zero in the image; the split-KV kernel puts each back to zero after
  // its merge)
  d.off_row_merge = off;
  off = align256(off + rows.size() * sizeof(MergeRef));
  d.off_combine_count = off;
  off = align256(off + combine.size() * sizeof(int32_t));
  d.n_stage_pages = (int32_t)stage_pages.size();
  d.off_stage_pages = off;
  off = align256(off + stage_pages.size() * sizeof(int32_t));
  d.off_stage_bt = off;
  off = align256(off + stage_bt.size() * sizeof(int32_t));
  d.metadata_bytes = off;
  d.off_part_lse = off;
  off = align256(off + (size_t)n_partials * sizeof(float));
  d.off_part_o = off;
  off = align256(off + (size_t)n_partials * D * sizeof(float));
  d.off_stage_kv = off;
  off = align256(off + 2 * stage_pages.size() * (size_t)Hkv * ps * D * 2);
  d.workspace_bytes = off;

  plan->host_image.assign(d.metadata_bytes, 0);
  uint8_t* img = plan->host_image.data();
  if (!items.empty())
    memcpy(img + d.off_decode_items, items.data(), items.size() * sizeof(DecodeItem));
  if (!rows.empty()) memcpy(img + d.off_rows, rows.data(), rows.size() * sizeof(RowDesc));
  if (!pitems.empty())
    memcpy(img + d.off_prefill_items, pitems.data(), pitems.size() * sizeof(PrefillItem));
  if (!combine.empty())
    memcpy(img + d.off_combine, combine.data(), combine.size() * sizeof(CombineEntry));
  if (!stage_pages.empty()) {
    memcpy(img + d.off_stage_pages, stage_pages.data(), stage_pages.size() * sizeof(int32_t));
    memcpy(img + d.off_stage_bt, stage_bt.data(), stage_bt.size() * sizeof(int32_t));
  }
  {
    std::vector<int32_t> slot_entry((size_t)n_partials, -1);
    for (size_t e = 0; e < combine.size(); ++e)
      for (int32_t k = 0; k < combine[e].n_slots; ++k)
        slot_entry[(size_t)combine[e].slot_begin + k] = (int32_t)e;
    MergeRef* mr = reinterpret_cast<MergeRef*>(img + d.off_row_merge);
    for (size_t i = 0; i < rows.size(); ++i) {
      MergeRef ref = {-1, 0, 0, 0};
      if (rows[i].dst >= 0) {
        const CombineEntry& ce = combine[(size_t)slot_entry[(size_t)rows[i].dst]];
        ref.entry = slot_entry[(size_t)rows[i].dst];
        ref.n_slots = ce.n_slots;
        ref.slot_begin = ce.slot_begin;
      }
      mr[i] = ref;
    }
  }

  mb_plan_info_t& info = plan->info;
  info = mb_plan_info_t{};
  info.n_decode_items = d.n_decode_items;
  info.n_decode_rows = d.n_decode_rows;
  info.n_prefill_items = d.n_prefill_items;
  info.n_combine = d.n_combine;
  info.n_partials = n_partials;
  info.n_cascade_groups = n_groups;
  info.cascade_keys = cascade_keys;
  info.kv_chunk = chunk;
  info.total_q = total_q;
  info.n_launches = (d.n_decode_items > 0) + (d.n_prefill_items > 0);
  info.workspace_bytes = d.workspace_bytes;
  info.metadata_bytes = d.metadata_bytes;
  info.prefill_ctas = d.prefill_ctas;
  info.staged_pages = d.n_stage_pages;
  info.splitkv_copies = d.decode_copies;
  info.splitkv_max_rows = d.decode_max_rows;
  return MB_OK;
}

// ---- pinned staging for the plan upload --------------------------------
// A copy from pageable memory makes the host wait for the stream's earlier
// work; the plan therefore uploads from page-locked buffers. Buffers are
// recycled once the event recorded after their copy has completed, so no
// call here blocks on the device.
namespace {
struct Staging {
  int device;
  void* ptr;
  size_t cap;
  cudaEvent_t done;
  bool in_use;
};
std::mutex g_staging_mu;
std::vector<Staging>* g_staging = new std::vector<Staging>();  // never freed: outlives exit
}  // namespace

int staging_acquire(int device, size_t bytes) {
  std::lock_guard<std::mutex> lk(g_staging_mu);
  for (size_t i = 0; i < g_staging->size(); ++i) {
    Staging& b = (*g_staging)[i];
    if (b.in_use || b.device != device || b.cap < bytes) continue;
    if (cudaEventQuery(b.done) != cudaSuccess) continue;
    b.in_use = true;
    return (int)i;
  }
  Staging b;
  b.device = device;
  b.cap = std::max<size_t>(bytes, 64 * 1024);
  if (cudaHostAlloc(&b.ptr, b.cap, cudaHostAllocDefault) != cudaSuccess) return -1;
  if (cudaEventCreateWithFlags(&b.done, cudaEventDisableTiming) != cudaSuccess) {
    cudaFreeHost(b.ptr);
    return -1;
  }
  b.in_use = true;
  g_staging->push_back(b);
  return (int)g_staging->size() - 1;
}

void* staging_ptr(int idx) {
  std::lock_guard<std::mutex> lk(g_staging_mu);
  return (*g_staging)[idx].ptr;
}

cudaError_t staging_record(int idx, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_staging_mu);
  return cudaEventRecord((*g_staging)[idx].done, s);
}

void staging_release(int idx) {
  std::lock_guard<std::mutex> lk(g_staging_mu);
  if (idx >= 0 && idx < (int)g_staging->size()) (*g_staging)[idx].in_use = false;
}

}  // namespace mb

extern "C" {

int32_t mb_abi_version(void) { return MB_ABI_VERSION; }

const char* mb_status_string(mb_status_t s) {
  switch (s) {
    case MB_OK: return "ok";
    case MB_ERR_INVALID_ARG: return "invalid argument";
    case MB_ERR_SHAPE: return "inconsistent shapes, triples or block table";
    case MB_ERR_UNSUPPORTED: return "unsupported head_dim / page_size / size";
    case MB_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case MB_ERR_CUDA: return "CUDA runtime error";
    case MB_ERR_TIMEOUT: return "a bounded device wait ran out";
    case MB_ERR_DEVICE_INDEX: return "device-side index out of range";
    case MB_ERR_SHARED_PAGE: return "a new row would be written into a shared page";
  }
  return "unknown status";
}

mb_status_t mb_slot_mapping(const mb_request_t* reqs, int32_t n_reqs,
                            const int32_t* block_table_host,
                            const mb_config_t* cfg, int32_t* slots_out,
                            int32_t total_q) {
  mb_status_t st = validate_config(cfg);
  if (st != MB_OK) return st;
  int32_t tq = 0;
  st = validate_requests(reqs, n_reqs, block_table_host, cfg, &tq);
  if (st != MB_OK) return st;
  if (total_q < tq || total_q < 0) return MB_ERR_SHAPE;
  if (total_q > 0 && !slots_out) return MB_ERR_INVALID_ARG;
  const int ps = cfg->page_size, mb = cfg->max_blocks_per_req;
  for (int32_t t = 0; t < total_q; ++t) slots_out[t] = -1;
  for (int32_t r = 0; r < n_reqs; ++r) {
    const mb_request_t& q = reqs[r];
    const int32_t s0 = q.kv_length - (q.q_end - q.q_start);
    for (int32_t t = q.q_start; t < q.q_end; ++t) {
      const int32_t p = s0 + (t - q.q_start);
      const int32_t page = block_table_host[(size_t)r * mb + p / ps];
      slots_out[t] = page * ps + p % ps;
    }
  }
  return MB_OK;
}

mb_status_t mb_check_append_targets(const mb_request_t* reqs, int32_t n_reqs,
                                    const int32_t* block_table_host, const mb_config_t* cfg,
                                    int32_t* bad_request_out) {
  if (bad_request_out) *bad_request_out = -1;
  mb_status_t st = validate_config(cfg);
  if (st != MB_OK) return st;
  int32_t tq = 0;
  st = validate_requests(reqs, n_reqs, block_table_host, cfg, &tq);
  if (st != MB_OK) return st;
  const int ps = cfg->page_size, mb = cfg->max_blocks_per_req;
  // how many requests map each page (a request mapping a page twice counts once)
  std::vector<int32_t> maps((size_t)cfg->num_pages, 0), last((size_t)cfg->num_pages, -1);
  for (int32_t r = 0; r < n_reqs; ++r) {
    const int32_t nb = (reqs[r].kv_length + ps - 1) / ps;
    for (int32_t b = 0; b < nb; ++b) {
      const int32_t page = block_table_host[(size_t)r * mb + b];
      if (last[(size_t)page] != r) {
        last[(size_t)page] = r;
        ++maps[(size_t)page];
      }
    }
  }
  for (int32_t r = 0; r < n_reqs; ++r) {
    const int32_t s0 = reqs[r].kv_length - (reqs[r].q_end - reqs[r].q_start);
    if (reqs[r].q_end == reqs[r].q_start) continue;
    for (int32_t b = s0 / ps; b <= (reqs[r].kv_length - 1) / ps; ++b) {
      if (maps[(size_t)block_table_host[(size_t)r * mb + b]] > 1) {
        if (bad_request_out) *bad_request_out = r;
        return MB_ERR_SHARED_PAGE;
      }
    }
  }
  return MB_OK;
}

mb_status_t mb_positions(const mb_request_t* reqs, int32_t n_reqs, int32_t* positions_out,
                         int32_t total_q) {
  if (n_reqs < 0 || total_q < 0) return MB_ERR_INVALID_ARG;
  if ((n_reqs > 0 && !reqs) || (total_q > 0 && !positions_out)) return MB_ERR_INVALID_ARG;
  for (int32_t t = 0; t < total_q; ++t) positions_out[t] = -1;
  for (int32_t r = 0; r < n_reqs; ++r) {
    const mb_request_t& q = reqs[r];
    if (q.q_start < 0 || q.q_end < q.q_start || q.q_end > total_q ||
        q.q_end - q.q_start > q.kv_length)
      return MB_ERR_SHAPE;
    const int32_t s0 = q.kv_length - (q.q_end - q.q_start);
    for (int32_t t = q.q_start; t < q.q_end; ++t) positions_out[t] = s0 + (t - q.q_start);
  }
  return MB_OK;
}

mb_status_t mb_attn_plan_ex(const mb_request_t* reqs, int32_t n_reqs,
                            const int32_t* block_table_host,
                            const mb_config_t* cfg,
                            const mb_plan_options_t* opts, void* workspace,
                            size_t* workspace_bytes, cudaStream_t stream,
                            mb_plan_t** out_plan) {
  if (!workspace_bytes) return MB_ERR_INVALID_ARG;
  mb_plan* plan = new (std::nothrow) mb_plan();
  if (!plan) return MB_ERR_INVALID_ARG;
  mb_status_t st = mb::build_plan(reqs, n_reqs, block_table_host, cfg, opts, plan);
  if (st != MB_OK) {
    delete plan;
    return st;
  }
  if (!workspace) {  // size query
    *workspace_bytes = plan->dev.workspace_bytes;
    delete plan;
    return MB_OK;
  }
  if (!out_plan) {
    delete plan;
    return MB_ERR_INVALID_ARG;
  }
  if (*workspace_bytes < plan->dev.workspace_bytes ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0) {
    delete plan;
    return MB_ERR_WORKSPACE;
  }
  plan->workspace = workspace;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) {
    delete plan;
    return MB_ERR_CUDA;
  }
  const size_t nb = plan->dev.metadata_bytes;
  plan->staging = mb::staging_acquire(device, nb);
  if (plan->staging < 0) {
    delete plan;
    return MB_ERR_CUDA;
  }
  memcpy(mb::staging_ptr(plan->staging), plan->host_image.data(), nb);
  cudaError_t e = cudaMemcpyAsync(workspace, mb::staging_ptr(plan->staging), nb,
                                  cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = mb::staging_record(plan->staging, stream);
  if (e != cudaSuccess) {
    mb::staging_release(plan->staging);
    delete plan;
    return MB_ERR_CUDA;
  }
  *out_plan = plan;
  return MB_OK;
}

mb_status_t mb_attn_plan(const mb_request_t* reqs, int32_t n_reqs,
                         const int32_t* block_table_host, const mb_config_t* cfg,
                         void* workspace, size_t* workspace_bytes,
                         cudaStream_t stream, mb_plan_t** out_plan) {
  return mb_attn_plan_ex(reqs, n_reqs, block_table_host, cfg, nullptr, workspace,
                         workspace_bytes, stream, out_plan);
}

mb_status_t mb_attn_plan_host(const mb_request_t* reqs, int32_t n_reqs,
                              const int32_t* block_table_host, const mb_config_t* cfg,
                              const mb_plan_options_t* opts, mb_plan_t** out_plan) {
  if (!out_plan) return MB_ERR_INVALID_ARG;
  mb_plan* plan = new (std::nothrow) mb_plan();
  if (!plan) return MB_ERR_INVALID_ARG;
  mb_status_t st = mb::build_plan(reqs, n_reqs, block_table_host, cfg, opts, plan);
  if (st != MB_OK) {
    delete plan;
    return st;
  }
  *out_plan = plan;
  return MB_OK;
}

mb_status_t mb_plan_export_metadata(const mb_plan_t* plan, void* dst, size_t dst_bytes) {
  if (!plan || !dst || dst_bytes < plan->host_image.size()) return MB_ERR_INVALID_ARG;
  memcpy(dst, plan->host_image.data(), plan->host_image.size());
  return MB_OK;
}

mb_status_t mb_plan_layout(const mb_plan_t* plan, size_t* out6) {
  if (!plan || !out6) return MB_ERR_INVALID_ARG;
  out6[0] = plan->dev.off_decode_items;
  out6[1] = plan->dev.off_rows;
  out6[2] = plan->dev.off_prefill_items;
  out6[3] = plan->dev.off_combine;
  out6[4] = plan->dev.off_part_lse;
  out6[5] = plan->dev.off_part_o;
  return MB_OK;
}

mb_status_t mb_plan_info(const mb_plan_t* plan, mb_plan_info_t* info) {
  if (!plan || !info) return MB_ERR_INVALID_ARG;
  *info = plan->info;
  return MB_OK;
}

mb_status_t mb_attn_destroy(mb_plan_t* plan) {
  if (plan && plan->staging >= 0) mb::staging_release(plan->staging);
  delete plan;
  return MB_OK;
}

}  // extern "C"
