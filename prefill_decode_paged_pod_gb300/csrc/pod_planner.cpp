// pod_planner.cpp — host-side POD planner.
//
// What the POD walkthrough's plan does ("plan 内部做了什么"): read the page
// tables on the host, derive each request's kv_len (get_seq_lens), and build
// the auxiliary structures every later run reuses. The batch wrapper plans the
// decode side first and decides from it how CTAs are shared with prefill
// ("Batch 版本 plan 的 colocated-CTA 调度细节", with the 1536-prefill-row cutoff).
//
// This planner does the same job for one persistent sm_103a launch:
//  1. validate both halves and compute kv_len / q_len;
//  2. cut prefill queries into 128-row tiles (ntok tokens x G qo heads of one
//     KV head) and trim each tile's key range by the causal diagonal and the
//     window;
//  3. cut decode queries into units of at most 32 rows and split each unit's
//     key range into chunks whose size is searched to balance the decode CTAs;
//  4. choose how many CTAs run prefill tiles and how many run decode items so
//     that both halves are predicted to finish together, and assign the work
//     with longest-processing-time-first list scheduling;
//  5. lay out the workspace: metadata (uploaded once) then split partials.
// Everything is a deterministic function of the inputs and num_sms. The
// schedule simulations run on integer times (1/256 ns), so they give the same
// result on every host; planning runs on the calling thread.
#include "pod_planner.hpp"

#include <algorithm>
#include <cstdlib>
#include <limits>
#include <cmath>
#include <cstring>
#include <functional>
#include <utility>

namespace {

constexpr int kInvalid = 1, kUnsupported = 2;

// ---- schedule arithmetic -----------------------------------------------------
// Simulated times are integers in 1/256 ns. A heap key packs a CTA's finish
// time and its index, (time << kCtaBits) | cta, so that comparing keys orders
// CTAs by finish time, then by index (the tie rule of every simulation here).
constexpr double kTicksPerNs = 256.0;
constexpr int kCtaBits = 20;                     // grids of up to 2^20 CTAs
constexpr uint64_t kCtaMask = (1ull << kCtaBits) - 1;
constexpr int64_t kNever = std::numeric_limits<int64_t>::max() >> (kCtaBits + 1);

int64_t ticks(double ns) { return (int64_t)std::llround(ns * kTicksPerNs); }
double ns_of(int64_t t) { return (double)t / kTicksPerNs; }
uint64_t key_of(int64_t t, int cta) { return ((uint64_t)t << kCtaBits) | (uint64_t)cta; }
int64_t time_of(uint64_t k) { return (int64_t)(k >> kCtaBits); }
int cta_of(uint64_t k) { return (int)(k & kCtaMask); }

// 4-ary min-heap of keys; the root is replaced in place (a CTA that takes a
// job finishes later and sinks).
struct KeyHeap {
  std::vector<uint64_t> k;
  // CTAs `ctas` (ascending) all free at time 0: ascending keys are a heap
  void reset(const std::vector<int>& ctas) {
    k.resize(ctas.size());
    for (size_t i = 0; i < ctas.size(); ++i) k[i] = key_of(0, ctas[i]);
  }
  void reset_range(int n) {
    k.resize((size_t)n);
    for (int i = 0; i < n; ++i) k[(size_t)i] = key_of(0, i);
  }
  uint64_t top() const { return k[0]; }
  void replace_top(uint64_t key) {
    uint64_t* a = k.data();
    const size_t n = k.size();
    size_t i = 0;
    for (;;) {
      const size_t c = 4 * i + 1;
      size_t m;
      uint64_t mk;
      if (c + 3 < n) {   // four children: pick the least without branches
        const size_t i01 = a[c + 1] < a[c] ? c + 1 : c;
        const size_t i23 = a[c + 3] < a[c + 2] ? c + 3 : c + 2;
        m = a[i23] < a[i01] ? i23 : i01;
        mk = a[m];
      } else {
        if (c >= n) break;
        m = c;
        mk = a[c];
        for (size_t j = c + 1; j < n; ++j)
          if (a[j] < mk) { mk = a[j]; m = j; }
      }
      if (mk >= key) break;
      a[i] = mk;
      i = m;
    }
    a[i] = key;
  }
};


// ---- cost model; constants measured on GB300 ------------------------------
// A CTA's speed depends on what shares its SM: the fused launch runs two CTAs
// per SM, and CTA c sits on SM c mod num_sms (the first num_sms CTAs take one
// slot of every SM, the next num_sms the second slot).
struct CostModel {
  double p_block_ns[3];  // one 64-key block of a 128-row tile; SM shared with
                         // [0] nothing, [1] a decode CTA, [2] another prefill CTA
  double p_tile_ns;      // per-tile setup + epilogue
  double p_flops_per_ns; // whole-GPU prefill ceiling
  double d_bytes_per_ns[3];  // decode stream of one CTA; SM shared with
                             // [0] nothing, [1] a prefill CTA, [2] another decode CTA
  double d_item_ns;      // per-item setup, pipeline fill and drain, output
  double hbm_bytes_per_ns;   // whole-GPU decode ceiling
};

CostModel cost_model(int d) {
  // Measured on GB300 with the c3-c5 workloads: per-CTA time of a 64-key
  // prefill block and per-CTA decode stream, by what shares the SM.
  CostModel c;
  const double f = 0.4 + 0.6 * d / 128.0;   // head_dim 64 halves the MMA work
  c.p_block_ns[0] = 800.0 * f;
  c.p_block_ns[1] = 1080.0 * f;
  c.p_block_ns[2] = 1150.0 * f;
  c.p_tile_ns = 1500.0;
  c.p_flops_per_ns = 1.2e6;
  c.d_bytes_per_ns[0] = 30.0;   // items of <= 16 rows; 32-row items cost 1.25x
  c.d_bytes_per_ns[1] = 24.0;
  c.d_bytes_per_ns[2] = 23.5;
  c.d_item_ns = 2500.0;
  c.hbm_bytes_per_ns = 7000.0;
  return c;
}

// Co-residency rates when most decode bytes are in items of more than 16
// rows (both mma m-tiles, all 8 decode warps busy): a timeline of the fused
// c5 launch on GB300 (per-record %globaltimer stamps) measured 17.1 GB/s for
// a decode CTA next to a prefill CTA against 19.3 GB/s next to a decode CTA,
// and prefill CTAs 1 % slower next to a decode CTA than next to another
// prefill CTA. Items of at most 16 rows leave half the decode warps idle and
// keep the rates above (measured best for c2-c4).
void wide_decode_neighbours(CostModel& c, int d) {
  const double f = 0.4 + 0.6 * d / 128.0;
  c.p_block_ns[1] = 1160.0 * f;
  c.d_bytes_per_ns[1] = c.d_bytes_per_ns[2] * (17.1 / 19.3);
}

// Co-residency class of CTA c (0 alone, 1 other role, 2 same role) when CTAs
// [0, n_p) run prefill and [n_p, n_p + n_d) decode, `cps` CTAs per SM.
int neighbour_class(int c, int n_p, int n_d, int S, int cps) {
  if (cps < 2) return 0;
  const int other = c < S ? c + S : c - S;
  if (other >= n_p + n_d) return 0;
  const bool me_p = c < n_p, other_p = other < n_p;
  return me_p == other_p ? 2 : 1;
}

int fail(std::string* err, int code, const std::string& msg) {
  if (err) *err = msg;
  return code;
}

int load_half(const char* name, const int32_t* q_indptr, const int32_t* kv_indptr,
              const int32_t* kv_indices, const int32_t* last, int batch, int num_pages, int ps,
              int causal, PodHalfHost& h, std::string* err) {
  std::string n(name);
  if (batch < 0) return fail(err, kInvalid, n + "_batch < 0");
  h.batch = batch;
  h.num_pages = num_pages;
  h.q_indptr.assign(1, 0);
  h.kv_indptr.assign(1, 0);
  h.kv_indices.clear();
  h.last_page_len.clear();
  h.kv_len.clear();
  h.q_len.clear();
  h.rows = 0;
  if (batch == 0) return 0;
  if (!q_indptr || !kv_indptr || !last)
    return fail(err, kInvalid, n + ": NULL page-table pointer for a non-empty half");
  if (q_indptr[0] != 0 || kv_indptr[0] != 0)
    return fail(err, kInvalid, n + ": q_indptr[0] and kv_indptr[0] must be 0");
  h.q_indptr.assign(q_indptr, q_indptr + batch + 1);
  h.kv_indptr.assign(kv_indptr, kv_indptr + batch + 1);
  h.last_page_len.assign(last, last + batch);
  for (int r = 0; r < batch; ++r) {
    if (q_indptr[r + 1] < q_indptr[r]) return fail(err, kInvalid, n + "_q_indptr is not monotone");
    if (kv_indptr[r + 1] < kv_indptr[r]) return fail(err, kInvalid, n + "_kv_indptr is not monotone");
  }
  int64_t npages_total = kv_indptr[batch];
  if (npages_total > 0) {
    if (!kv_indices) return fail(err, kInvalid, n + "_kv_indices is NULL");
    h.kv_indices.assign(kv_indices, kv_indices + npages_total);
    for (int64_t i = 0; i < npages_total; ++i)
      if (kv_indices[i] < 0 || kv_indices[i] >= num_pages)
        return fail(err, kInvalid, n + "_kv_indices[" + std::to_string(i) + "] = " +
                                       std::to_string(kv_indices[i]) + " is outside the page pool of " +
                                       std::to_string(num_pages));
  }
  h.kv_len.resize(batch);
  h.q_len.resize(batch);
  for (int r = 0; r < batch; ++r) {
    int64_t ql = (int64_t)q_indptr[r + 1] - q_indptr[r];
    int64_t np = (int64_t)kv_indptr[r + 1] - kv_indptr[r];
    int64_t kl = 0;
    if (np > 0) {
      if (last[r] < 1 || last[r] > ps)
        return fail(err, kInvalid, n + "_last_page_len[" + std::to_string(r) + "] = " +
                                       std::to_string(last[r]) + " is outside [1, page_size]");
      kl = (np - 1) * (int64_t)ps + last[r];
    }
    if (kl > INT32_MAX) return fail(err, kInvalid, n + ": kv_len overflows int32");
    if (ql > 0 && kl == 0)
      return fail(err, kInvalid, n + ": request " + std::to_string(r) + " has queries but no keys");
    if (ql > 0 && causal && kl < ql)
      return fail(err, kInvalid, n + ": request " + std::to_string(r) +
                                     " has kv_len < q_len under the causal mask");
    h.kv_len[r] = (int32_t)kl;
    h.q_len[r] = (int32_t)ql;
  }
  h.rows = q_indptr[batch];
  return 0;
}

// Key range [lo, hi) needed by the query tokens [t0, t0 + ntok) of a request:
// bottom-right diagonal p = kv_len - q_len + i, window keeps t >= p - window_left.
void key_range(int kv_len, int q_len, int t0, int ntok, int causal, int window_left, int* lo,
               int* hi) {
  int64_t p_first = (int64_t)kv_len - q_len + t0;
  int64_t p_last = p_first + ntok - 1;
  int64_t h = kv_len;
  if (causal) h = std::min<int64_t>(kv_len, p_last + 1);
  int64_t l = 0;
  if (window_left >= 0) l = std::max<int64_t>(0, p_first - window_left);
  if (l > h) l = h;
  *lo = (int)l;
  *hi = (int)h;
}

int64_t nblocks(int lo, int hi) {
  int64_t b0 = (int64_t)(lo / POD_KBLOCK) * POD_KBLOCK;
  return (hi - b0 + POD_KBLOCK - 1) / POD_KBLOCK;
}

// The makespan of longest-processing-time-first list scheduling on CTAs of
// different speeds: jobs, given in decreasing size, go to the CTA that would
// finish them first. `work` is in work units, `rate[c]` units per ns,
// `overhead` ns per job. CTAs of equal rate form one class (a heap on finish
// time, ties to the lowest index), so a job costs one probe per class.
// Returns the makespan (ns); stops as soon as it reaches `bound` and returns
// that time.
struct RateClasses {
  std::vector<double> rate;
  std::vector<KeyHeap> heap;
  void build(const std::vector<double>& r) {
    rate.clear();
    heap.clear();
    std::vector<std::vector<int>> members;
    for (int c = 0; c < (int)r.size(); ++c) {
      size_t k = 0;
      while (k < rate.size() && rate[k] != r[c]) ++k;
      if (k == rate.size()) {
        rate.push_back(r[c]);
        members.emplace_back();
      }
      members[k].push_back(c);
    }
    heap.resize(rate.size());
    for (size_t k = 0; k < rate.size(); ++k) heap[k].reset(members[k]);
  }
};

double lpt_makespan(const std::vector<double>& sorted_work, double overhead,
                    const std::vector<double>& rate, double bound) {
  if (rate.empty() || sorted_work.empty()) return 0.0;
  RateClasses cl;
  cl.build(rate);
  const int64_t tb = std::isinf(bound) ? kNever : ticks(bound);
  int64_t makespan = 0;
  for (double w : sorted_work) {
    int best = -1;
    uint64_t bk = 0;
    for (size_t k = 0; k < cl.rate.size(); ++k) {
      const uint64_t top = cl.heap[k].top();
      const uint64_t cand = key_of(time_of(top) + ticks(overhead + w / cl.rate[k]), cta_of(top));
      if (best < 0 || cand < bk) { best = (int)k; bk = cand; }
    }
    makespan = std::max(makespan, time_of(bk));
    if (makespan >= tb) return ns_of(makespan);
    cl.heap[best].replace_top(bk);
  }
  return ns_of(makespan);
}

// What-if simulations run on a scaled copy of a schedule: every `s`
// consecutive jobs of a list sorted by decreasing cost become one job of
// their mean cost (the total work is kept), and every `s`-th CTA stands for
// its group. A makespan then takes about 1/s of the heap operations; it
// stays comparable across the candidates a search weighs. s is the largest
// power of two up to 8 that divides the CTA count and leaves at least 1024
// jobs.
int sim_scale(size_t jobs, int ctas) {
  int s = 1;
  while (s < 8 && ctas % (2 * s) == 0 && jobs / (size_t)(2 * s) >= 1024) s *= 2;
  return s;
}
std::vector<double> scaled_jobs(const std::vector<double>& sorted, int s) {
  if (s <= 1) return sorted;
  std::vector<double> out;
  out.reserve(sorted.size() / s + 1);
  for (size_t i = 0; i < sorted.size(); i += (size_t)s) {
    const size_t e = std::min(sorted.size(), i + (size_t)s);
    double sum = 0.0;
    for (size_t j = i; j < e; ++j) sum += sorted[j];
    out.push_back(sum / (double)s);
  }
  return out;
}

struct DecodeUnit {
  int req, kv_head, tok0, ntok, lo, hi;
};

// Split [lo, hi) into ceil(len / chunk) nearly equal chunks with inner
// boundaries on multiples of 64 keys.
void split_range(int lo, int hi, int chunk, std::vector<std::pair<int, int>>& out) {
  out.clear();
  int64_t len = hi - lo;
  if (chunk <= 0 || len <= chunk) {
    out.push_back({lo, hi});
    return;
  }
  int64_t n = (len + chunk - 1) / chunk;
  int prev = lo;
  for (int64_t j = 1; j < n; ++j) {
    int64_t b = lo + (j * len) / n;
    b = (b / POD_DECODE_STAGE) * POD_DECODE_STAGE;
    if (b <= prev || b >= hi) continue;
    out.push_back({prev, (int)b});
    prev = (int)b;
  }
  out.push_back({prev, hi});
}

struct DecodeChoice {
  double time = 0.0;
  int chunk = 0;
};

// bytes of K/V a decode item streams: keys x 2 rows (K, V) x d x 2 bytes
double item_bytes(int keys, int d) { return 4.0 * d * (double)keys; }
// scheduling weight of a decode item: its bytes, times 1.25 when its rows
// fill two mma m-tiles (more compute per byte streamed)
double item_work(int keys, int d, int rows) {
  return item_bytes(keys, d) * (rows > 16 ? 1.25 : 1.0);
}

// Estimated decode time (ns) with key chunks of `chunk` (0 = no split). When
// even the bandwidth floor plus the split's cost reaches `bound`, that lower
// bound is returned without scheduling the items.
double decode_time(const std::vector<DecodeUnit>& units, const std::vector<double>& rate,
                   int chunk, int G, int d, const CostModel& cm, double total_bytes,
                   double bound = std::numeric_limits<double>::infinity()) {
  // item counts by key count, for items of <= 16 rows ([0]) and more ([1])
  int max_keys = 0;
  for (const DecodeUnit& u : units) max_keys = std::max(max_keys, u.hi - u.lo);
  // Capacity bound: over a makespan T, CTA c does at most rate[c] * (T -
  // overhead * its items) work, so T >= (work + items * overhead * r_min) /
  // sum(rate). Splitting keeps the total work (an item's work is linear in
  // its keys) and only adds items, so the bound with one item per unit, plus
  // the merge launch a split plan pays, holds before any item is built.
  double r_min = std::numeric_limits<double>::infinity(), r_sum = 0.0;
  for (double r : rate) {
    r_min = std::min(r_min, r);
    r_sum += r;
  }
  // A unit longer than the chunk splits into ceil(len / chunk) parts (inner
  // boundaries are at least chunk - 64 >= 192 keys apart for the chunks
  // searched, so none coincide): the item count and the partial rows' bytes
  // are known before any item is built.
  if (chunk > 0 && !std::isinf(bound) && r_sum > 0.0) {
    double w = 0.0, items = 0.0, sbytes = 0.0;
    for (const DecodeUnit& u : units) {
      const int len = u.hi - u.lo;
      w += item_work(len, d, u.ntok * G);
      const int n = len > chunk ? (len + chunk - 1) / chunk : 1;
      items += n;
      if (n > 1) sbytes += (double)n * u.ntok * G * (d + 1) * 4.0 * 2.0;
    }
    const double ex = sbytes > 0 ? 8000.0 + sbytes / cm.hbm_bytes_per_ns : 0.0;
    const double lb = std::max(total_bytes / cm.hbm_bytes_per_ns + ex,
                               (w + items * cm.d_item_ns * r_min) / r_sum + ex);
    if (lb >= bound) return lb;
  }
  std::vector<int> cnt[2] = {std::vector<int>(max_keys + 1, 0), std::vector<int>(max_keys + 1, 0)};
  std::vector<std::pair<int, int>> parts;
  double split_bytes = 0.0;
  size_t n_items = 0;
  for (const DecodeUnit& u : units) {
    split_range(u.lo, u.hi, chunk, parts);
    const int f = u.ntok * G > 16 ? 1 : 0;
    for (auto& pr : parts) ++cnt[f][pr.second - pr.first];
    n_items += parts.size();
    if (parts.size() > 1) split_bytes += (double)parts.size() * u.ntok * G * (d + 1) * 4.0 * 2.0;
  }
  // splitting costs the partial rows' round trip and the merge launch
  const double extra = split_bytes > 0 ? 8000.0 + split_bytes / cm.hbm_bytes_per_ns : 0.0;
  const double floor_t = total_bytes / cm.hbm_bytes_per_ns + extra;
  if (floor_t >= bound) return floor_t;
  // the capacity bound again, with the items this chunk makes
  if (r_sum > 0.0) {
    double w = 0.0;
    for (int f = 0; f < 2; ++f)
      for (int k = 0; k <= max_keys; ++k)
        if (cnt[f][k]) w += cnt[f][k] * item_work(k, d, f ? 32 : 16);
    const double lb = (w + (double)n_items * cm.d_item_ns * r_min) / r_sum + extra;
    if (lb >= bound) return lb;
  }
  // only the makespan is needed and equal jobs are interchangeable: the work
  // values in decreasing order (the order lpt's index sort gives), merged
  // from the two count tables
  std::vector<double> work;
  work.reserve(n_items);
  int k0 = max_keys, k1 = max_keys;
  for (;;) {
    while (k0 >= 0 && cnt[0][k0] == 0) --k0;
    while (k1 >= 0 && cnt[1][k1] == 0) --k1;
    if (k0 < 0 && k1 < 0) break;
    const double w0 = k0 >= 0 ? item_work(k0, d, 16) : -1.0;
    const double w1 = k1 >= 0 ? item_work(k1, d, 32) : -1.0;
    if (w0 >= w1) {
      work.insert(work.end(), cnt[0][k0], w0);
      cnt[0][k0] = 0;
    } else {
      work.insert(work.end(), cnt[1][k1], w1);
      cnt[1][k1] = 0;
    }
  }
  const int sc = sim_scale(work.size(), (int)rate.size());
  std::vector<double> srate;
  for (size_t c = 0; c < rate.size(); c += (size_t)sc) srate.push_back(rate[c]);
  // a scaled job stands for `sc` jobs: its per-job overhead is theirs, shared
  double t = lpt_makespan(scaled_jobs(work, sc), cm.d_item_ns, srate, bound - extra);
  t = std::max(t, total_bytes / cm.hbm_bytes_per_ns);
  return t + extra;
}

// Items and partial rows a chunk makes (a unit longer than the chunk splits
// into ceil(len / chunk) parts, each writing R = ntok * G partial rows).
void chunk_counts(const std::vector<DecodeUnit>& units, int chunk, int G, int64_t* items,
                  int64_t* prows) {
  *items = 0;
  *prows = 0;
  for (const DecodeUnit& u : units) {
    const int len = u.hi - u.lo;
    const int64_t n = (chunk > 0 && len > chunk) ? (len + chunk - 1) / chunk : 1;
    *items += n;
    if (n > 1) *prows += n * u.ntok * G;
  }
}

// The decode chunk with the least estimated time; with limits (>= 0), only
// chunks whose items and partial rows fit them (no split always does).
DecodeChoice best_decode(const std::vector<DecodeUnit>& units, const std::vector<double>& rate,
                         int G, int d, const CostModel& cm, double total_bytes,
                         int64_t max_items = -1, int64_t max_prows = -1) {
  DecodeChoice best;
  // 0 = no split; then 16 Ki .. 256 keys. A candidate at or above the longest
  // key range splits nothing and is the unsplit plan again: skipped.
  const int cands[] = {0, 16384, 8192, 4096, 2048, 1024, 512, 256};
  int max_keys = 0;
  for (const DecodeUnit& u : units) max_keys = std::max(max_keys, u.hi - u.lo);
  best.time = decode_time(units, rate, 0, G, d, cm, total_bytes);
  best.chunk = 0;
  for (int c : cands) {
    if (c == 0 || c >= max_keys) continue;
    if (max_items >= 0) {
      int64_t it, pr;
      chunk_counts(units, c, G, &it, &pr);
      if (it > max_items || pr > max_prows) continue;
    }
    // taken only below best * (1 - 1e-9): no simulation needs to run past that
    const double t = decode_time(units, rate, c, G, d, cm, total_bytes, best.time * (1.0 - 1e-9));
    if (t < best.time * (1.0 - 1e-9)) {
      best.time = t;
      best.chunk = c;
    }
  }
  return best;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Keys per TMA box for the half's K/V, or 0 when page boxes do not fit the
// page table (then the kernel gathers with cp.async). page_size >= 8 (a power
// of two): one page (at most 64 slots) per box. page_size 1, 2, 4: the longest
// run of 64, 32, 16 or 8 keys such that every aligned run of that many keys of
// every request lies on consecutive pages, so one box covers kbx / ps pages.
int tma_box_keys(const PodHalfHost& h, int ps) {
  if (ps <= 0 || (ps & (ps - 1)) != 0 || ps > 256) return 0;
  if (ps >= 8) return ps < 64 ? ps : 64;
  for (int kbx = 64; kbx >= 8; kbx /= 2) {
    const int n = kbx / ps;  // pages per box
    bool ok = true;
    for (int r = 0; r < h.batch && ok; ++r) {
      const int base = h.kv_indptr[r], np = h.kv_indptr[r + 1] - h.kv_indptr[r];
      for (int g0 = 0; g0 < np && ok; g0 += n) {
        const int m = std::min(n, np - g0);
        for (int i = 1; i < m; ++i)
          if (h.kv_indices[base + g0 + i] != h.kv_indices[base + g0] + i) { ok = false; break; }
      }
    }
    if (ok) return kbx;
  }
  return 0;
}

}  // namespace

int pod_build_plan(const PodPlanArgs& a, PodPlanHost& P, std::string* err) {
  if (a.H <= 0 || a.Hk <= 0) return fail(err, kInvalid, "num_qo_heads and num_kv_heads must be positive");
  if (a.H % a.Hk != 0)
    return fail(err, kInvalid, "num_qo_heads must be a multiple of num_kv_heads");
  if (a.ps <= 0) return fail(err, kInvalid, "page_size must be positive");
  if (a.d != 64 && a.d != 128 && a.d != 256)
    return fail(err, kUnsupported, "head_dim must be 64, 128 or 256");
  if (a.d == 256 && a.rope)
    return fail(err, kUnsupported, "RoPE with head_dim 256");
  if (a.dtype != 0 && a.dtype != 1) return fail(err, kUnsupported, "dtype must be fp16 or bf16");
  if (a.window_left < -1) return fail(err, kInvalid, "window_left must be -1 or >= 0");
  if (a.num_sms <= 0) return fail(err, kInvalid, "num_sms must be positive");
  const int G = a.H / a.Hk;
  if (G > POD_TILE_ROWS) return fail(err, kUnsupported, "more than 128 qo heads per kv head");

  P.H = a.H; P.Hk = a.Hk; P.G = G; P.d = a.d; P.ps = a.ps;
  P.causal = a.causal ? 1 : 0; P.window_left = a.window_left;
  P.p_custom_mask = a.p_custom_mask ? 1 : 0;
  P.rope = a.rope ? 1 : 0;
  P.rope_scale = a.rope_scale;
  P.rope_theta = a.rope_theta;
  if (P.rope && (!(a.rope_scale > 0.0) || !(a.rope_theta > 0.0) || !std::isfinite(a.rope_scale) ||
                 !std::isfinite(a.rope_theta)))
    return fail(err, kInvalid, "rope_scale and rope_theta must be finite and positive");
  P.dtype = a.dtype; P.has_sinks = a.has_sinks ? 1 : 0; P.num_sms = a.num_sms;
  P.sm_scale = a.sm_scale > 0.f ? a.sm_scale : (float)(1.0 / std::sqrt((double)a.d));
  P.scale_log2 = (float)((double)P.sm_scale * 1.4426950408889634);

  int rc = load_half("p", a.p_q_indptr, a.p_kv_indptr, a.p_kv_indices, a.p_last_page_len,
                     a.p_batch, a.p_num_pages, a.ps, P.causal, P.p, err);
  if (rc) return rc;
  rc = load_half("d", a.d_q_indptr, a.d_kv_indptr, a.d_kv_indices, a.d_last_page_len, a.d_batch,
                 a.d_num_pages, a.ps, P.causal, P.dd, err);
  if (rc) return rc;
  if (P.dd.rows > 0 && G > POD_DECODE_ROWS)
    return fail(err, kUnsupported, "more than 32 qo heads per kv head on the decode half");
  // The RoPE kernel holds the low parts of the rotated operands and the
  // head_dim 256 kernel a 256-column O (TMEM) and 224 KB of stages: they run
  // one CTA per SM; the others two.
  const int cps = (P.rope || a.d > 128) ? 1 : POD_CTAS_PER_SM;
  P.ctas_per_sm = cps;

  // CUDA-graph capacity mode (POD walkthrough, "CUDAGraph 模式的运行时约束":
  // a fixed batch and page-table buffers reserved at their maximum size,
  // with plan run outside capture): every table is laid out for the
  // capacities, the grid is the full grid, and this plan must fit them.
  P.graph = a.graph ? 1 : 0;
  if (P.graph) {
    if (P.rope || P.p_custom_mask)
      return fail(err, kUnsupported, "CUDA-graph capacity with RoPE or a custom prefill mask");
    const int caps[6] = {a.cap_p_batch, a.cap_p_rows, a.cap_p_pages,
                         a.cap_d_batch, a.cap_d_rows, a.cap_d_pages};
    for (int c : caps)
      if (c < 0) return fail(err, kInvalid, "capacities must be >= 0");
    const PodHalfHost* hh[2] = {&P.p, &P.dd};
    const char* nm[2] = {"prefill", "decode"};
    for (int k = 0; k < 2; ++k) {
      const int64_t pages = hh[k]->kv_indptr.back();
      if (hh[k]->batch > caps[3 * k] || hh[k]->rows > caps[3 * k + 1] || pages > caps[3 * k + 2])
        return fail(err, kInvalid, std::string(nm[k]) + " half exceeds its capacity: " +
                                       std::to_string(hh[k]->batch) + " requests, " +
                                       std::to_string(hh[k]->rows) + " rows, " +
                                       std::to_string(pages) + " pages against " +
                                       std::to_string(caps[3 * k]) + ", " +
                                       std::to_string(caps[3 * k + 1]) + ", " +
                                       std::to_string(caps[3 * k + 2]));
    }
    P.cap_p_batch = a.cap_p_batch; P.cap_p_rows = a.cap_p_rows; P.cap_p_pages = a.cap_p_pages;
    P.cap_d_batch = a.cap_d_batch; P.cap_d_rows = a.cap_d_rows; P.cap_d_pages = a.cap_d_pages;
  }

  CostModel cm = cost_model(a.d);

  // ---- decode units ---------------------------------------------------------
  const int Tu = std::max(1, POD_DECODE_ROWS / G);
  P.tu = Tu;
  // under RoPE the prefill half reads compact copies through an identity
  // page table; the decode half reads the caller's cache
  auto identity_half = [](const PodHalfHost& h) {
    PodHalfHost c = h;
    for (size_t i = 0; i < c.kv_indices.size(); ++i) c.kv_indices[i] = (int32_t)i;
    return c;
  };
  P.p_tma = tma_box_keys(P.rope ? identity_half(P.p) : P.p, a.ps);
  // decode boxes hold both 64-element halves of head_dim; they are laid out
  // for page_size >= 8 (a page per box) and 1 (runs of pages) only
  P.d_tma = (a.ps == 1 || a.ps >= 8) ? tma_box_keys(P.dd, a.ps) : 0;
  // in capacity mode the load path may not depend on the page tables: page
  // boxes for page_size >= 8, the cp.async gather below
  if (P.graph) {
    P.p_tma = a.ps >= 8 ? P.p_tma : 0;
    P.d_tma = a.ps >= 8 ? P.d_tma : 0;
  }
  std::vector<DecodeUnit> units;
  double d_bytes = 0.0, d_bytes_wide = 0.0;
  for (int r = 0; r < P.dd.batch; ++r) {
    int ql = P.dd.q_len[r], kl = P.dd.kv_len[r];
    for (int t0 = 0; t0 < ql; t0 += Tu) {
      int nt = std::min(Tu, ql - t0);
      int lo, hi;
      key_range(kl, ql, t0, nt, P.causal, P.window_left, &lo, &hi);
      for (int g = 0; g < P.Hk; ++g) {
        units.push_back({r, g, t0, nt, lo, hi});
        d_bytes += 4.0 * a.d * (double)(hi - lo);
        if (nt * G > 16) d_bytes_wide += 4.0 * a.d * (double)(hi - lo);
      }
    }
  }
  if (d_bytes_wide > 0.5 * d_bytes) wide_decode_neighbours(cm, a.d);

  // ---- prefill tiles --------------------------------------------------------
  // A tile's key range is split into chunks (merged like decode splits) when
  // the prefill half is small enough to share SMs with split CTAs: at most
  // 1536 query rows, the batch plan's cutoff for colocated prefill CTAs
  // (POD walkthrough, "Batch 版本 plan 的 colocated-CTA 调度细节"), too few
  // tiles to give every CTA of the grid one, and a longest tile that would
  // outlast the balanced makespan of both halves. Next to a long decode
  // stream (c4) the tiles already finish early; a split there only adds the
  // merge.
  const int Tq = std::max(1, POD_TILE_ROWS / G);
  const int grid_cap = a.num_sms * cps;
  struct TileUnit { int r, g, t0, nt, lo, hi; };
  std::vector<TileUnit> tunits;
  for (int r = 0; r < P.p.batch; ++r) {
    int ql = P.p.q_len[r], kl = P.p.kv_len[r];
    for (int t0 = 0; t0 < ql; t0 += Tq) {
      int nt = std::min(Tq, ql - t0);
      int lo, hi;
      key_range(kl, ql, t0, nt, P.causal && !P.p_custom_mask, P.window_left, &lo, &hi);
      for (int g = 0; g < P.Hk; ++g) tunits.push_back({r, g, t0, nt, lo, hi});
    }
  }
  int p_split = 1;
  if (!P.graph && P.p.rows <= 1536 && !tunits.empty() && 2 * (int)tunits.size() <= grid_cap) {
    double longest = 0.0, total = 0.0;
    for (const TileUnit& u : tunits) {
      const double t = cm.p_tile_ns + (double)nblocks(u.lo, u.hi) * cm.p_block_ns[2];
      longest = std::max(longest, t);
      total += t;
    }
    for (const DecodeUnit& u : units)
      total += cm.d_item_ns + item_work(u.hi - u.lo, a.d, u.ntok * G) / cm.d_bytes_per_ns[2];
    if (longest > total / grid_cap)
      p_split = (grid_cap + (int)tunits.size() - 1) / (int)tunits.size();
  }
  P.ptiles.clear();
  std::vector<int32_t> pgroups;
  std::vector<int32_t> pgroup_rows;
  std::vector<double> tile_cost;
  double p_flops = 0.0;
  int p_prows = 0;
  {
    std::vector<std::pair<int, int>> parts;
    for (const TileUnit& u : tunits) {
      const int len = u.hi - u.lo;
      // chunks of at least 8 key blocks, 64-key aligned inside the range
      const int n = std::max(1, std::min(p_split, len / (8 * POD_KBLOCK)));
      const int chunk = n > 1 ? ((len + n - 1) / n + POD_KBLOCK - 1) / POD_KBLOCK * POD_KBLOCK : 0;
      split_range(u.lo, u.hi, chunk, parts);
      const int R = u.nt * G;
      int prow0 = -1;
      if (parts.size() > 1) {
        prow0 = p_prows;
        p_prows += (int)parts.size() * R;
        int32_t grp[POD_REC] = {0, u.r, u.g, u.t0, u.nt, prow0, (int)parts.size(), R};
        pgroups.insert(pgroups.end(), grp, grp + POD_REC);
        pgroup_rows.push_back(R);
      }
      for (size_t j = 0; j < parts.size(); ++j) {
        const int prow = prow0 < 0 ? -1 : prow0 + (int)j * R;
        int32_t rec[POD_REC] = {u.r, u.g, u.t0, u.nt, parts[j].first, parts[j].second, prow, 0};
        P.ptiles.insert(P.ptiles.end(), rec, rec + POD_REC);
        tile_cost.push_back((double)nblocks(parts[j].first, parts[j].second));
      }
      p_flops += 4.0 * a.d * (double)u.nt * G * (double)len;
    }
  }
  const int n_tiles = (int)tile_cost.size();
  P.tq = Tq;

  // ---- CTA split between the halves ----------------------------------------
  const int S = a.num_sms;
  const int grid_max = S * cps;
  // capacity mode: table sizes from the capacities alone. A request of q
  // rows makes ceil(q / t) token blocks of each kv head; splits may add up to
  // one item per CTA, and the partial rows of split items are bounded.
  int64_t cap_tiles = 0, cap_units = 0, cap_items = 0, cap_prows = 0;
  if (P.graph) {
    cap_tiles = ((int64_t)(P.cap_p_rows + Tq - 1) / Tq + P.cap_p_batch) * P.Hk;
    cap_units = ((int64_t)(P.cap_d_rows + Tu - 1) / Tu + P.cap_d_batch) * P.Hk;
    cap_items = cap_units + grid_max;
    cap_prows = (int64_t)2 * grid_max * POD_DECODE_ROWS;
  }
  // per-CTA rates for a split: prefill in blocks per ns, decode in bytes per ns
  auto rates = [&](int n_p, int n_d, std::vector<double>& rp, std::vector<double>& rd) {
    rp.resize(n_p);
    rd.resize(n_d);
    for (int c = 0; c < n_p; ++c) rp[c] = 1.0 / cm.p_block_ns[neighbour_class(c, n_p, n_d, S, cps)];
    for (int c = 0; c < n_d; ++c)
      rd[c] = cm.d_bytes_per_ns[neighbour_class(n_p + c, n_p, n_d, S, cps)];
  };
  int n_p = 0;
  int chunk = 0;
  if (n_tiles > 0 && units.empty()) {
    n_p = std::min(grid_max, n_tiles);
  } else if (!units.empty()) {
    // decode chunk size for the decode share of the CTAs, estimated from the
    // total CTA-time of each half at same-role rates
    double p_total = 0.0, d_total = 0.0;
    for (double b : tile_cost) p_total += cm.p_tile_ns + b * cm.p_block_ns[2];
    for (const DecodeUnit& u : units)
      d_total += cm.d_item_ns + item_work(u.hi - u.lo, a.d, u.ntok * G) / cm.d_bytes_per_ns[2];
    n_p = n_tiles > 0 ? (int)std::lround(grid_max * p_total / (p_total + d_total)) : 0;
    n_p = std::min(std::max(n_p, n_tiles > 0 ? 1 : 0), std::min(grid_max - 1, n_tiles));
    std::vector<double> rp, rd;
    rates(n_p, grid_max - n_p, rp, rd);
    chunk = best_decode(units, rd, G, a.d, cm, d_bytes, P.graph ? cap_items : -1,
                        P.graph ? cap_prows : -1).chunk;
  }
  int n_d_max = grid_max - n_p;
  // The kernel serves both queues to every CTA, so the split only sets where
  // each CTA starts. Choose it on a simulation of the two queues: long
  // prefill tiles that start late can set the makespan (c4: 128 tiles of 128
  // blocks against 256 long decode requests).
  if (n_tiles > 0 && !units.empty()) {
    std::vector<double> tile_ns(tile_cost.size());
    for (size_t t = 0; t < tile_cost.size(); ++t) tile_ns[t] = tile_cost[t];
    std::sort(tile_ns.begin(), tile_ns.end(), std::greater<double>());
    std::vector<double> item_b;
    std::vector<std::pair<int, int>> parts;
    for (const DecodeUnit& u : units) {
      split_range(u.lo, u.hi, chunk, parts);
      for (auto& pr : parts) item_b.push_back(item_work(pr.second - pr.first, a.d, u.ntok * G));
    }
    std::sort(item_b.begin(), item_b.end(), std::greater<double>());
    // Makespan when CTAs [0, np) start on tiles and the rest on items: a CTA
    // takes the next job of its own queue when free, the other queue's once
    // its own is empty; CTAs are served in (finish time, index) order. Job
    // costs are precomputed for each co-residency class. The simulation stops
    // as soon as a CTA's finish time reaches `bound` (the candidate can no
    // longer win) and returns that time.
    const double floor_t = std::max(p_flops / cm.p_flops_per_ns, d_bytes / cm.hbm_bytes_per_ns);
    // the simulations run scaled by sc (sc CTAs, sc jobs per simulated one)
    const int sc = sim_scale(tile_ns.size() + item_b.size(), S);
    const std::vector<double> tile_s = scaled_jobs(tile_ns, sc), item_s = scaled_jobs(item_b, sc);
    const int S_s = S / sc, grid_s = grid_max / sc;
    std::vector<int64_t> tile_t[3], item_t[3];
    for (int k = 0; k < 3; ++k) {
      tile_t[k].resize(tile_s.size());
      item_t[k].resize(item_s.size());
      for (size_t t = 0; t < tile_s.size(); ++t)
        tile_t[k][t] = ticks(cm.p_tile_ns + tile_s[t] * cm.p_block_ns[k]);
      for (size_t t = 0; t < item_s.size(); ++t)
        item_t[k][t] = ticks(cm.d_item_ns + item_s[t] / cm.d_bytes_per_ns[k]);
    }
    KeyHeap heap;
    std::vector<int> cls(grid_s);
    auto queue_makespan = [&](int np, double bound) -> double {
      if (floor_t >= bound) return floor_t;
      const int64_t tb = std::isinf(bound) ? kNever : ticks(bound);
      for (int c = 0; c < grid_s; ++c) cls[c] = neighbour_class(c, np, grid_s - np, S_s, cps);
      heap.reset_range(grid_s);
      const size_t nt = tile_s.size(), ni = item_s.size();
      size_t it = 0, id = 0;
      int64_t makespan = 0;
      while (it < nt || id < ni) {
        const uint64_t top = heap.top();
        const int c = cta_of(top);
        const bool want_p = c < np ? it < nt : id >= ni;
        const int64_t tn = time_of(top) + (want_p ? tile_t[cls[c]][it++] : item_t[cls[c]][id++]);
        makespan = std::max(makespan, tn);
        if (makespan >= tb) return ns_of(makespan);
        heap.replace_top(key_of(tn, c));
      }
      return std::max(ns_of(makespan), floor_t);
    };
    const int hi_np = std::min(grid_max - 1, n_tiles);
    const int hi_s = std::max(1, std::min(grid_s - 1, (hi_np + sc - 1) / sc));
    const int np0_s = std::max(1, std::min(hi_s, (n_p + sc / 2) / sc));
    const double share_t = queue_makespan(np0_s, std::numeric_limits<double>::infinity());
    int best_np = np0_s;
    double best_t = share_t;
    // Golden-section search of the split over [1, hi_s] (the makespan is
    // close to unimodal in it: too few prefill-first CTAs start long tiles
    // late, too many starve the decode stream), then the last few points.
    // Every simulation runs against the best time so far, which it can only
    // beat by more than 1e-9 to be taken.
    std::vector<double> seen(hi_s + 2, -1.0);
    auto eval = [&](int np) -> double {
      if (seen[np] < 0.0) {
        seen[np] = np == np0_s ? share_t : queue_makespan(np, best_t * (1.0 - 1e-9));
        if (seen[np] < best_t * (1.0 - 1e-9)) { best_t = seen[np]; best_np = np; }
      }
      return seen[np];
    };
    {
      const double phi = 0.6180339887498949;
      int lo = 1, hi = hi_s;
      int x1 = hi - (int)std::lround(phi * (hi - lo)), x2 = lo + (int)std::lround(phi * (hi - lo));
      while (hi - lo > 3) {
        if (x1 >= x2) x2 = x1 + 1;
        if (eval(x1) <= eval(x2)) {
          hi = x2;
          x2 = x1;
          x1 = hi - (int)std::lround(phi * (hi - lo));
        } else {
          lo = x1;
          x1 = x2;
          x2 = lo + (int)std::lround(phi * (hi - lo));
        }
      }
      for (int np = lo; np <= hi; ++np) eval(np);
    }
    best_np = best_np == np0_s ? n_p : std::min(hi_np, best_np * sc);
    // the model is coarse: leave the balanced split unless the queues are
    // predicted to finish at least 1 % earlier another way
    if (best_t < 0.99 * share_t) n_p = best_np;
    n_d_max = grid_max - n_p;
  }

  // ---- decode items, partial rows, merge groups -------------------------------
  P.ditems.clear();
  P.mgroups = pgroups;      // prefill merge groups first, then decode ones
  P.mrow_ptr.assign(1, 0);
  for (int R : pgroup_rows) P.mrow_ptr.push_back(P.mrow_ptr.back() + R);
  std::vector<double> item_cost;
  int n_prows = p_prows;
  std::vector<std::pair<int, int>> parts;
  for (const DecodeUnit& u : units) {
    split_range(u.lo, u.hi, chunk, parts);
    const int R = u.ntok * G;
    int prow0 = -1;
    if (parts.size() > 1) {
      prow0 = n_prows;
      n_prows += (int)parts.size() * R;
      int32_t g[POD_REC] = {1, u.req, u.kv_head, u.tok0, u.ntok, prow0, (int)parts.size(), R};
      P.mgroups.insert(P.mgroups.end(), g, g + POD_REC);
      P.mrow_ptr.push_back(P.mrow_ptr.back() + R);
    }
    for (size_t j = 0; j < parts.size(); ++j) {
      int prow = prow0 < 0 ? -1 : prow0 + (int)j * R;
      int32_t rec[POD_REC] = {u.req, u.kv_head, u.tok0, u.ntok, parts[j].first, parts[j].second,
                              prow, 0};
      P.ditems.insert(P.ditems.end(), rec, rec + POD_REC);
      item_cost.push_back(item_work(parts[j].second - parts[j].first, a.d, R));
    }
  }
  const int n_items = (int)item_cost.size();
  // decode-first CTAs beyond the item count still pay off while there are
  // prefill tiles left for them (they go straight to that queue); no more
  // CTAs than jobs
  int n_d = std::min(n_d_max, std::max(n_items, n_tiles + n_items - n_p));
  if (n_items == 0) n_d = 0;
  // capacity mode: the launch shape may not depend on the plan, so the grid
  // is always full (CTAs that find both queues empty leave at once)
  if (P.graph) n_d = grid_max - n_p;
  P.n_p_ctas = n_p;
  P.n_d_ctas = n_d;
  P.grid = n_p + n_d;
  P.decode_chunk = chunk;
  P.n_prows = n_prows;
  P.n_mrows = P.mrow_ptr.back();

  // ---- work queues and per-CTA lists ------------------------------------------
  // The kernel's queues hold every tile / item in decreasing cost (ties by
  // index). The per-CTA lists deal each queue round-robin over the CTAs that
  // start on it: what each CTA would take if all ran at one speed. The kernel
  // serves the queues; the lists are kept for inspection.
  P.cta_ptr.assign(P.grid + 1, 0);
  P.cta_list.clear();
  {
    auto order_of = [](const std::vector<double>& cost) {
      std::vector<int> idx(cost.size());
      for (size_t i = 0; i < idx.size(); ++i) idx[i] = (int)i;
      std::stable_sort(idx.begin(), idx.end(), [&](int a, int b) { return cost[a] > cost[b]; });
      return idx;
    };
    std::vector<std::vector<int>> lists(P.grid);
    P.pqueue.clear();
    P.dqueue.clear();
    if (n_p > 0) {
      P.pqueue = order_of(tile_cost);
      for (size_t k = 0; k < P.pqueue.size(); ++k) lists[k % (size_t)n_p].push_back(P.pqueue[k]);
    }
    if (n_d > 0) {
      P.dqueue = order_of(item_cost);
      for (size_t k = 0; k < P.dqueue.size(); ++k)
        lists[n_p + k % (size_t)n_d].push_back(P.dqueue[k]);
    }
    P.dqrec.clear();
    P.dqrec.reserve(P.dqueue.size() * POD_DQREC);
    for (int j : P.dqueue) {
      const int32_t* rec = &P.ditems[(size_t)j * POD_REC];
      const int r = rec[0];
      P.dqrec.insert(P.dqrec.end(), rec, rec + POD_REC);
      const int32_t ext[POD_DQREC - POD_REC] = {P.dd.kv_len[r], P.dd.q_indptr[r], P.dd.q_len[r],
                                               P.dd.kv_indptr[r],
                                               P.dd.kv_indptr[r + 1] - P.dd.kv_indptr[r], 0, 0, 0};
      P.dqrec.insert(P.dqrec.end(), ext, ext + POD_DQREC - POD_REC);
    }
    P.cta_list.reserve(P.pqueue.size() + P.dqueue.size());
    for (int c = 0; c < P.grid; ++c) {
      P.cta_ptr[c] = (int32_t)P.cta_list.size();
      P.cta_list.insert(P.cta_list.end(), lists[c].begin(), lists[c].end());
    }
    P.cta_ptr[P.grid] = (int32_t)P.cta_list.size();
  }

  // ---- custom-mask bit offsets: request r's [q_len, kv_len] bits start after
  // those of the requests before it
  P.p_mask_off.clear();
  P.p_mask_bits = 0;
  if (P.p_custom_mask) {
    int64_t bit = 0;
    for (int r = 0; r <= P.p.batch; ++r) {
      P.p_mask_off.push_back((int32_t)(uint32_t)((uint64_t)bit & 0xffffffffu));
      P.p_mask_off.push_back((int32_t)(uint32_t)((uint64_t)bit >> 32));
      if (r < P.p.batch) bit += (int64_t)P.p.q_len[r] * P.p.kv_len[r];
    }
    P.p_mask_bits = bit;
  }

  // ---- RoPE pre-pass tables: per prefill page-table entry the position of
  // slot 0 and the slots below kv_len; per query row of either half its
  // bottom-right position. The cos/sin table covers every key position of
  // both halves (decode keys are rotated in the kernel) and every |query
  // position|.
  P.p_rope_ent.clear(); P.d_rope_ent.clear(); P.p_rope_qpos.clear(); P.d_rope_qpos.clear();
  P.rope_rows = 0;
  if (P.rope) {
    int64_t rows = 1;
    auto tables = [&](const PodHalfHost& h, std::vector<int32_t>* ent, std::vector<int32_t>& qpos) {
      for (int r = 0; r < h.batch; ++r) {
        const int np = h.kv_indptr[r + 1] - h.kv_indptr[r];
        for (int i = 0; i < np && ent; ++i) {
          ent->push_back(i * P.ps);
          ent->push_back(std::max(0, std::min(P.ps, h.kv_len[r] - i * P.ps)));
        }
        rows = std::max<int64_t>(rows, (int64_t)np * P.ps);
        for (int i = 0; i < h.q_len[r]; ++i) {
          const int64_t pos = (int64_t)h.kv_len[r] - h.q_len[r] + i;
          qpos.push_back((int32_t)pos);
          rows = std::max<int64_t>(rows, (pos < 0 ? -pos : pos) + 1);
        }
      }
    };
    tables(P.p, &P.p_rope_ent, P.p_rope_qpos);
    tables(P.dd, nullptr, P.d_rope_qpos);
    P.rope_rows = (int)rows;
  }

  // ---- workspace layout -----------------------------------------------------------
  size_t off = 0;
  auto place = [&](size_t n_int32) {
    size_t o = off;
    off = align_up(off + std::max<size_t>(n_int32, 1) * 4, 16);
    return o;
  };
  // capacity mode: every table at its capacity (this plan fits: checked
  // above for the page tables, by construction for the rest)
  auto sz = [&](size_t actual, int64_t capacity) -> size_t {
    return P.graph ? (size_t)std::max<int64_t>(capacity, (int64_t)actual) : actual;
  };
  if (P.graph && ((int64_t)n_tiles > cap_tiles || (int64_t)n_items > cap_items ||
                  (int64_t)n_prows > cap_prows || (int64_t)P.n_mrows > cap_prows))
    return fail(err, kInvalid, "plan exceeds the capacity layout");
  P.cap_mrows = P.graph ? (int)cap_prows : P.n_mrows;
  P.cap_tiles = P.graph ? (int)cap_tiles : n_tiles;
  P.cap_items = P.graph ? (int)cap_items : n_items;
  P.off_status = place(64);
  P.off_p_q_indptr = place(sz(P.p.q_indptr.size(), (int64_t)P.cap_p_batch + 1));
  P.off_p_kv_indptr = place(sz(P.p.kv_indptr.size(), (int64_t)P.cap_p_batch + 1));
  P.off_p_kv_indices = place(sz(P.p.kv_indices.size(), P.cap_p_pages));
  P.off_p_kv_len = place(sz(P.p.kv_len.size(), P.cap_p_batch));
  P.off_d_q_indptr = place(sz(P.dd.q_indptr.size(), (int64_t)P.cap_d_batch + 1));
  P.off_d_kv_indptr = place(sz(P.dd.kv_indptr.size(), (int64_t)P.cap_d_batch + 1));
  P.off_d_kv_indices = place(sz(P.dd.kv_indices.size(), P.cap_d_pages));
  P.off_d_kv_len = place(sz(P.dd.kv_len.size(), P.cap_d_batch));
  P.off_ptiles = place(sz(P.ptiles.size(), cap_tiles * POD_REC));
  P.off_ditems = place(sz(P.ditems.size(), cap_items * POD_REC));
  P.off_cta_ptr = place(sz(P.cta_ptr.size(), (int64_t)grid_max + 1));
  P.off_cta_list = place(sz(P.cta_list.size(), cap_tiles + cap_items));
  P.off_mgroups = place(sz(P.mgroups.size(), cap_units * POD_REC));
  P.off_mrow_ptr = place(sz(P.mrow_ptr.size(), cap_units + 1));
  P.off_pqueue = place(sz(P.pqueue.size(), cap_tiles));
  P.off_dqueue = place(sz(P.dqueue.size(), cap_items));
  P.off_dqrec = place(sz(P.dqrec.size(), cap_items * POD_DQREC));
  P.off_p_mask_off = place(P.p_mask_off.size());
  if (P.rope) {
    P.off_p_rope_src = place(P.p.kv_indices.size());
    P.off_p_rope_ent = place(P.p_rope_ent.size());
    P.off_p_rope_qpos = place(P.p_rope_qpos.size());
    P.off_d_rope_qpos = place(P.d_rope_qpos.size());
  }
  P.int_bytes = align_up(off, 256);
  P.off_part_o = P.int_bytes;
  const size_t prows_sz = sz((size_t)n_prows, cap_prows);
  P.off_part_lse = align_up(P.off_part_o + prows_sz * a.d * 4, 256);
  size_t end = align_up(P.off_part_lse + std::max<size_t>(prows_sz, 1) * 4, 256);
  if (P.rope) {
    // cos/sin table [rows][d/2] (float2), then the prefill page copies
    // (rows K_hi, V, K_lo: 16-bit) and the high and low parts of the rotated
    // queries of both halves
    const size_t page_bytes = (size_t)3 * P.ps * P.Hk * a.d * 2;
    P.off_rope_table = end;
    end = align_up(end + (size_t)P.rope_rows * (a.d / 2) * 8, 256);
    P.off_p_kvcopy = end;
    end = align_up(end + P.p.kv_indices.size() * page_bytes, 256);
    const size_t pq = (size_t)P.p.rows * P.H * a.d * 2, dq = (size_t)P.dd.rows * P.H * a.d * 2;
    P.off_p_qcopy = end;
    end = align_up(end + pq, 256);
    P.off_p_qcopy_lo = end;
    end = align_up(end + pq, 256);
    P.off_d_qcopy = end;
    end = align_up(end + dq, 256);
    P.off_d_qcopy_lo = end;
    end = align_up(end + dq, 256);
  }
  P.total_bytes = end;

  P.int_image.assign(P.int_bytes, 0);
  auto put = [&](size_t o, const std::vector<int32_t>& v) {
    if (!v.empty()) std::memcpy(P.int_image.data() + o, v.data(), v.size() * 4);
  };
  {
    int32_t* st = reinterpret_cast<int32_t*>(P.int_image.data() + P.off_status);
    st[POD_ST_NTILES] = n_tiles;
    st[POD_ST_NITEMS] = n_items;
    st[POD_ST_NPCTAS] = P.n_p_ctas;
    st[POD_ST_NGROUPS] = (int32_t)(P.mgroups.size() / POD_REC);
    st[POD_ST_NMROWS] = P.n_mrows;
  }
  put(P.off_p_q_indptr, P.p.q_indptr);
  put(P.off_p_kv_indptr, P.p.kv_indptr);
  std::vector<int32_t> ident;
  auto identity = [&](size_t n) -> const std::vector<int32_t>& {
    ident.resize(n);
    for (size_t i = 0; i < n; ++i) ident[i] = (int32_t)i;
    return ident;
  };
  put(P.off_p_kv_indices, P.rope ? identity(P.p.kv_indices.size()) : P.p.kv_indices);
  put(P.off_p_kv_len, P.p.kv_len);
  put(P.off_d_q_indptr, P.dd.q_indptr);
  put(P.off_d_kv_indptr, P.dd.kv_indptr);
  put(P.off_d_kv_indices, P.dd.kv_indices);
  put(P.off_d_kv_len, P.dd.kv_len);
  put(P.off_ptiles, P.ptiles);
  put(P.off_ditems, P.ditems);
  put(P.off_cta_ptr, P.cta_ptr);
  put(P.off_cta_list, P.cta_list);
  put(P.off_mgroups, P.mgroups);
  put(P.off_mrow_ptr, P.mrow_ptr);
  put(P.off_pqueue, P.pqueue);
  put(P.off_dqueue, P.dqueue);
  put(P.off_dqrec, P.dqrec);
  // capacity mode: the kernels serve the queues up to their capacities, so
  // every position past the plan's own records is a sentinel (tile -1, a
  // decode record of request -1)
  if (P.graph) {
    int32_t* pq = reinterpret_cast<int32_t*>(P.int_image.data() + P.off_pqueue);
    for (int i = n_tiles; i < P.cap_tiles; ++i) pq[i] = -1;
    int32_t* dq = reinterpret_cast<int32_t*>(P.int_image.data() + P.off_dqrec);
    for (int i = n_items; i < P.cap_items; ++i) dq[(size_t)i * POD_DQREC] = -1;
  }
  put(P.off_p_mask_off, P.p_mask_off);
  if (P.rope) {
    put(P.off_p_rope_src, P.p.kv_indices);
    put(P.off_p_rope_ent, P.p_rope_ent);
    put(P.off_p_rope_qpos, P.p_rope_qpos);
    put(P.off_d_rope_qpos, P.d_rope_qpos);
  }

  P.summary.assign(S_COUNT, 0);
  int32_t* s = P.summary.data();
  s[S_H] = P.H; s[S_HK] = P.Hk; s[S_D] = P.d; s[S_PS] = P.ps; s[S_CAUSAL] = P.causal;
  s[S_WINDOW] = P.window_left; s[S_DTYPE] = P.dtype; s[S_SINKS] = P.has_sinks;
  s[S_NUM_SMS] = P.num_sms; s[S_GRID] = P.grid; s[S_NP_CTAS] = P.n_p_ctas;
  s[S_ND_CTAS] = P.n_d_ctas; s[S_NTILES] = n_tiles; s[S_NITEMS] = n_items;
  s[S_NGROUPS] = (int32_t)(P.mgroups.size() / POD_REC); s[S_NMROWS] = P.n_mrows;
  s[S_NPROWS] = P.n_prows; s[S_P_ROWS] = P.p.rows; s[S_D_ROWS] = P.dd.rows;
  s[S_P_BATCH] = P.p.batch; s[S_D_BATCH] = P.dd.batch; s[S_DECODE_CHUNK] = chunk;
  s[S_WS_LO] = (int32_t)(P.total_bytes & 0x7fffffff);
  s[S_WS_HI] = (int32_t)(P.total_bytes >> 31);
  s[S_P_TMA] = P.p_tma;
  s[S_D_TMA] = P.d_tma;
  s[S_P_MASK] = P.p_custom_mask;
  s[S_ROPE] = P.rope;
  return 0;
}
