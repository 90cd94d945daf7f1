// Host-side layout packing and mask-aware tile planning for MIS attention.
//
// The mask is eq. (4) of "From Generation to Scoring: Scaling LLM-Based
// Semantic Labeling at LinkedIn" (Section 4.1): with Q the shared rows and
// I_i the rows of item i (both contiguous, disjoint), key k is visible from
// row j iff k <= j and (k in Q or j, k in the same I_i). Because every set is
// contiguous, the visible keys of row j are at most two intervals:
//     [s0, min(pend, j+1))  and  [lo(j), j]
// where lo(j) is the first row of the set holding j (s0 for rows of Q). The
// planner walks 128-row query tiles and lists only the key tiles that meet
// one of those intervals for some row of the tile, so fully masked tiles cost
// neither FLOPs nor bytes (both pages skip tiles with no visible entry:
// Section 4.2 of "From Generation to Scoring", and "Turbocharging LinkedIn's
// recommendation systems with SGLang", section "FlashInfer changes").
#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>

#include "mis_internal.h"

namespace mis {

namespace {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Cost of a unit in softmax-step units (one step: two 128x128 S tiles, one
// per stream, with their PV products); a masked tile costs 5/4 of a full one.
// kUnitCost covers a unit's Q load, the turn-around of its first and last
// tiles and the hand-over of O to the epilogue warps. Fitted on GB300 as
// time = fixed + step * makespan to kernel times of both schedules on eleven
// packed batches (single requests of 3.5K to 19.5K rows, 16 to 640 requests
// of up to 555K rows in all): a unit costs one step; every unit cost between
// 0.5 and 1.5 steps picks the faster schedule on all of them. The split
// schedule's doubled K/V tile loads show up in that per-unit cost rather than
// in a per-step factor.
constexpr double kUnitCost = 1.0;

// Largest per-block total of unit costs when `units` (in list order, each
// repeated `reps` times for its heads) are dealt to min(total, n_blocks)
// persistent blocks in the kernel's snake order.
double snake_makespan(const std::vector<double>& cost, int reps, int n_blocks) {
  const int64_t total = (int64_t)cost.size() * reps;
  if (total == 0) return 0.0;
  const int64_t G = std::min<int64_t>(total, n_blocks);
  thread_local std::vector<double> load;
  load.assign((size_t)G, 0.0);
  // walk position u = kk * G + i runs through the units in list order; unit u
  // is list entry u / reps, tracked without a division
  int64_t q = 0, r = 0;
  for (int64_t kk = 0; kk * G < total; ++kk)
    for (int64_t i = 0; i < G && kk * G + i < total; ++i) {
      const int64_t c = (kk & 1) ? (G - 1 - i) : i;
      load[(size_t)c] += cost[(size_t)q];
      if (++r == reps) { r = 0; ++q; }
    }
  return *std::max_element(load.begin(), load.end());
}

// A query tile while the plan is built: its key-tile list and its costs.
struct Tmp { int32_t req, q0, kofs, nk; int64_t cost, cost_even, cost_odd; int64_t order; };

// Shared tail of both planners: unit order, schedule, statistics and the
// workspace layout. `T` is the row count seg_start covers.
mis_status_t finish_plan(HostPlan* p, std::vector<Tmp>& tmp, int32_t B, int32_t T,
                         int64_t visible, int64_t causal_tiles);

}  // namespace

mis_status_t build_plan(const mis_attn_desc* d, HostPlan* p) {
  if (!d || !p) return MIS_ERR_INVALID_ARG;
  if (d->B < 1 || d->T < 1 || d->Hq < 1 || d->Hkv < 1) return MIS_ERR_INVALID_ARG;
  if (!d->cu_seqlens || !d->prefix_len) return MIS_ERR_INVALID_ARG;
  if (d->Hq % d->Hkv) return MIS_ERR_SHAPE;
  if (d->D != 64 && d->D != 128) return MIS_ERR_UNSUPPORTED;
  if (!(d->scale >= 0.f) || std::isinf(d->scale)) return MIS_ERR_INVALID_ARG;
  // the grid is (query tiles) x Hq blocks and the key-tile flag uses bit 31
  if ((int64_t)d->T * d->Hq > (int64_t)1 << 40) return MIS_ERR_SHAPE;

  const int32_t B = d->B, T = d->T;
  const int32_t* cu = d->cu_seqlens;
  if (cu[0] != 0 || cu[B] != T) return MIS_ERR_SHAPE;
  for (int b = 0; b < B; ++b)
    if (cu[b + 1] <= cu[b]) return MIS_ERR_SHAPE;

  p->B = B; p->T = T; p->Hq = d->Hq; p->Hkv = d->Hkv; p->D = d->D;
  p->scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt((float)d->D);
  p->req.assign(B, ReqInfo{});
  p->seg_start.assign(T, 0);
  p->work.clear(); p->klist.clear(); p->tile_map.clear();
  p->stats = mis_plan_stats{};

  // ---- sets Q and I_i: validate and record lo(j) for every row ----
  for (int b = 0; b < B; ++b) {
    const int32_t s0 = cu[b], e0 = cu[b + 1], S = d->prefix_len[b];
    if (S < 1 || S > e0 - s0) return MIS_ERR_SHAPE;
    const int32_t pend = s0 + S;
    p->req[b] = ReqInfo{s0, e0, pend, 0};
    std::fill(p->seg_start.begin() + s0, p->seg_start.begin() + pend, s0);
    int32_t i0 = 0, i1 = 0;
    if (d->item_ptr) {
      i0 = d->item_ptr[b]; i1 = d->item_ptr[b + 1];
      if (i0 < 0 || i1 < i0 || (b == 0 && i0 != 0)) return MIS_ERR_SHAPE;
      if (i1 > i0 && !d->item_offsets) return MIS_ERR_INVALID_ARG;
    }
    // visible pairs: row j of Q sees [s0, j]; row d of an item set of n rows
    // sees the S rows of Q and d + 1 rows of its own set
    p->stats.visible_pairs += (int64_t)S * (S + 1) / 2;
    if (i1 == i0) {
      if (pend != e0) return MIS_ERR_SHAPE;      // rows after Q would belong to no set
      continue;
    }
    if (d->item_offsets[i0] != pend) return MIS_ERR_SHAPE;
    for (int32_t i = i0; i < i1; ++i) {
      const int32_t a = d->item_offsets[i];
      const int32_t e = (i + 1 < i1) ? d->item_offsets[i + 1] : e0;
      if (a < pend || e <= a || e > e0) return MIS_ERR_SHAPE;
      std::fill(p->seg_start.begin() + a, p->seg_start.begin() + e, a);
      const int64_t n = e - a;
      p->stats.visible_pairs += n * S + n * (n + 1) / 2;
    }
  }

  // ---- tiles ----
  // per-thread scratch: keeps its capacity from plan to plan
  thread_local std::vector<Tmp> tmp;
  tmp.clear();
  int64_t visible = 0, causal_tiles = 0;
  {
    // exact sizes first (the same interval arithmetic as below), so the lists
    // are filled without reallocation
    size_t n_tiles = 0, n_qt = 0;
    for (int b = 0; b < B; ++b) {
      const ReqInfo& R = p->req[b];
      const int32_t nqt = (R.e0 - R.s0 + kBM - 1) / kBM;
      n_qt += (size_t)nqt;
      for (int32_t t = 0; t < nqt; ++t) {
        const int32_t r0 = R.s0 + t * kBM, r1 = std::min(r0 + kBM, R.e0);
        const int32_t qb = (std::min(R.pend, r1) - R.s0 + kBN - 1) / kBN;
        const int32_t ba = (p->seg_start[r0] - R.s0) / kBN, bb = (r1 - 1 - R.s0) / kBN + 1;
        n_tiles += (size_t)qb + (size_t)std::max(0, bb - std::max(ba, qb));
      }
    }
    tmp.reserve(n_qt);
    p->klist.resize(n_tiles);
    p->tile_map.resize(4 * n_tiles);
  }
  visible = p->stats.visible_pairs;
  uint32_t* kl = p->klist.data();
  int32_t* tm = p->tile_map.data();
  int32_t n_emitted = 0, n_full = 0;
  for (int b = 0; b < B; ++b) {
    const ReqInfo& R = p->req[b];
    const int32_t L = R.e0 - R.s0;
    const int32_t nqt = (L + kBM - 1) / kBM;
    for (int32_t t = 0; t < nqt; ++t) {
      const int32_t r0 = R.s0 + t * kBM;
      const int32_t r1 = std::min(r0 + kBM, R.e0);
      causal_tiles += ((r1 - 1 - R.s0) / kBN) + 1;
      const int32_t lo_min = p->seg_start[r0];       // lo(j) never decreases with j
      const int32_t lo_max = p->seg_start[r1 - 1];
      // interval 1: keys of Q up to the last row; interval 2: [lo_min, r1)
      const int32_t qa = 0, qb = (std::min(R.pend, r1) - R.s0 + kBN - 1) / kBN;  // [qa, qb)
      const int32_t ba = (lo_min - R.s0) / kBN, bb = (r1 - 1 - R.s0) / kBN + 1;  // [ba, bb)
      Tmp w{b, r0, n_emitted, 0, 0, 0, 0, (int64_t)tmp.size()};
      auto emit = [&](int32_t u) {
        const int32_t c0 = R.s0 + u * kBN;
        const int32_t c1 = std::min(c0 + kBN, R.e0);
        // full iff every (j in [r0,r1), k in [c0,c1)) is visible:
        //   causal part: c1 - 1 <= r0;
        //   set part: keys at or past pend must be >= lo(j) for every row.
        const bool full = (c1 - 1 <= r0) && (c1 <= R.pend || std::max(c0, R.pend) >= lo_max);
        // a clipped key tile loads rows of the next request: mask it too
        const bool need_mask = !full || (c0 + kBN > R.e0);
        kl[n_emitted] = (uint32_t)c0 | (need_mask ? kNeedMask : 0u);
        int32_t* q = tm + 4 * (size_t)n_emitted;
        q[0] = b; q[1] = t; q[2] = u; q[3] = full ? 1 : 2;
        ++n_emitted;
        n_full += full ? 1 : 0;
        const int c = need_mask ? 5 : 4;   // masked tiles spend extra ALU in the softmax
        (w.nk % 2 ? w.cost_odd : w.cost_even) += c;
        ++w.nk;
        w.cost += c;
      };
      for (int32_t u = qa; u < qb; ++u) emit(u);
      for (int32_t u = std::max(ba, qb); u < bb; ++u) emit(u);
      tmp.push_back(w);
    }
  }
  if ((size_t)n_emitted != p->klist.size()) return MIS_ERR_SHAPE;   // the pre-count is exact
  p->stats.n_full = n_full;
  p->stats.n_partial = n_emitted - n_full;
  return finish_plan(p, tmp, B, T, visible, causal_tiles);
}

namespace {

mis_status_t finish_plan(HostPlan* p, std::vector<Tmp>& tmp, int32_t B, int32_t T,
                         int64_t visible, int64_t causal_tiles) {
  if (p->klist.size() > (size_t)std::numeric_limits<int32_t>::max()) return MIS_ERR_SHAPE;
  // Order: request by request, requests with the most expensive query tile
  // first, and inside a request the query tiles longest first. Blocks that run
  // at the same time then work on the same request and share its K/V tiles
  // through L2 (a request-blind longest-first order scatters them and every
  // query tile re-reads its request's K/V from HBM), while the long units
  // still start first.
  std::vector<int64_t> req_max(B, 0);
  for (const Tmp& w : tmp) req_max[w.req] = std::max(req_max[w.req], w.cost);
  {
    // the same order as a stable sort by (heaviest tile of the request
    // descending, request, tile cost descending), as one sort of packed keys:
    // request rank | inverted cost | list index
    thread_local std::vector<int32_t> rank, pos_of;
    thread_local std::vector<uint64_t> key;
    thread_local std::vector<Tmp> sorted;
    rank.resize((size_t)B);
    for (int b = 0; b < B; ++b) rank[(size_t)b] = b;
    std::stable_sort(rank.begin(), rank.end(),
                     [&](int32_t a, int32_t b) { return req_max[(size_t)a] > req_max[(size_t)b]; });
    pos_of.resize((size_t)B);
    for (int b = 0; b < B; ++b) pos_of[(size_t)rank[(size_t)b]] = b;
    int64_t cmax = 0;
    for (const Tmp& w : tmp) cmax = std::max(cmax, w.cost);
    if (cmax >= ((int64_t)1 << 24) || tmp.size() >= ((size_t)1 << 24) || B >= (1 << 16))
      return MIS_ERR_SHAPE;
    key.resize(tmp.size());
    for (size_t i = 0; i < tmp.size(); ++i)
      key[i] = ((uint64_t)pos_of[(size_t)tmp[i].req] << 48) |
               ((uint64_t)(((int64_t)1 << 24) - 1 - tmp[i].cost) << 24) | (uint64_t)i;
    std::sort(key.begin(), key.end());
    sorted.clear();
    sorted.reserve(tmp.size());
    for (uint64_t k : key) sorted.push_back(tmp[(size_t)(k & 0xFFFFFFu)]);
    tmp.swap(sorted);
  }
  p->work.reserve(tmp.size());
  for (const Tmp& w : tmp) p->work.push_back(WorkItem{w.req, w.q0, w.kofs, w.nk});

  // ---- schedule: head pairs, or one head with the key tiles split between
  // the two softmax streams. Pairs need an even GQA group; otherwise the one
  // with the smaller snake makespan over the device's SMs.
  const bool even_group = (p->Hq / p->Hkv) % 2 == 0;
  bool split = !even_group;
  const int32_t forced = schedule_override();
  if (even_group && forced == MIS_SCHEDULE_SPLIT) {
    split = true;
  } else if (even_group && forced == MIS_SCHEDULE_AUTO && !tmp.empty()) {
    thread_local std::vector<double> c_pair, c_split;
    c_pair.clear();
    c_split.clear();
    for (const Tmp& w : tmp) {
      c_pair.push_back(w.cost / 4.0 + kUnitCost);
      c_split.push_back(std::max(w.cost_even, w.cost_odd) / 4.0 + kUnitCost);
    }
    const int sms = num_sms();
    split = snake_makespan(c_split, p->Hq, sms) < snake_makespan(c_pair, p->Hq / 2, sms);
  }
  p->split = split;
  p->n_head_groups = split ? p->Hq : p->Hq / 2;
  p->stats.schedule = split ? MIS_SCHEDULE_SPLIT : MIS_SCHEDULE_PAIR;
  p->stats.n_units = (int64_t)p->work.size() * p->n_head_groups;

  // ---- unit order: the snake walk over the list, or, when the blocks come
  // out clearly better balanced, a wave-by-wave longest-processing-time
  // assignment: pass k still hands out the list's units kG..kG+G-1 (so blocks
  // that run together work on neighbouring units and share a request's K/V
  // tiles through L2), but the longest of them go to the blocks with the
  // least work so far. Laid out on the kernel's walk positions.
  p->order.clear();
  {
    const int64_t n_units = p->stats.n_units;
    const int64_t G = std::min<int64_t>(n_units, num_sms());
    if (n_units > G && G > 0 && n_units < ((int64_t)1 << 30)) {
      // costs in quarter steps (exact: tile costs are 4 or 5 quarters, a
      // unit costs kUnitCost more), so loads compare as integers
      const int64_t unit_q = (int64_t)(4.0 * kUnitCost);
      thread_local std::vector<int64_t> cost, load;
      thread_local std::vector<double> costd;
      thread_local std::vector<uint64_t> ukey, bkey;
      cost.resize((size_t)n_units);
      costd.resize((size_t)n_units);
      for (int64_t u = 0; u < n_units; ++u) {
        const Tmp& w = tmp[(size_t)(u / p->n_head_groups)];
        cost[(size_t)u] = (split ? std::max(w.cost_even, w.cost_odd) : w.cost) + unit_q;
        costd[(size_t)u] = cost[(size_t)u] / 4.0;
      }
      const double snake = snake_makespan(costd, 1, (int)G);
      const int64_t passes = (n_units + G - 1) / G;
      std::vector<int32_t>& order = p->order;      // laid out here, kept if it wins
      order.assign((size_t)(passes * G), -1);
      load.assign((size_t)G, 0);
      bkey.resize((size_t)G);
      thread_local std::vector<int32_t> uord, bord, cnt;
      uord.resize((size_t)G);
      bord.resize((size_t)G);
      // Stable counting sort of n values v(i) (i ascending within equal values)
      // into `out`, ascending or descending; false when their range is too
      // wide for it (the caller then sorts packed keys).
      auto counting = [&](int64_t n, auto v, bool descending, std::vector<int32_t>& out) -> bool {
        int64_t lo = v(0), hi = v(0);
        for (int64_t i = 1; i < n; ++i) { lo = std::min(lo, v(i)); hi = std::max(hi, v(i)); }
        if (hi - lo >= 4096) return false;
        cnt.assign((size_t)(hi - lo + 2), 0);
        for (int64_t i = 0; i < n; ++i) ++cnt[(size_t)((descending ? hi - v(i) : v(i) - lo) + 1)];
        for (size_t k = 1; k < cnt.size(); ++k) cnt[k] += cnt[k - 1];
        for (int64_t i = 0; i < n; ++i)
          out[(size_t)cnt[(size_t)(descending ? hi - v(i) : v(i) - lo)]++] = (int32_t)i;
        return true;
      };
      bool fits = true;
      for (int64_t kk = 0; kk < passes && fits; ++kk) {
        const int64_t u0 = kk * G, u1 = std::min(u0 + G, n_units), nu = u1 - u0;
        // units of the pass: cost descending, then list order
        if (!counting(nu, [&](int64_t i) { return cost[(size_t)(u0 + i)]; }, true, uord)) {
          ukey.resize((size_t)nu);
          for (int64_t i = 0; i < nu; ++i)
            ukey[(size_t)i] = ((uint64_t)(((int64_t)1 << 31) - 1 - cost[(size_t)(u0 + i)]) << 32) |
                              (uint64_t)i;
          std::sort(ukey.begin(), ukey.end());
          for (int64_t i = 0; i < nu; ++i) uord[(size_t)i] = (int32_t)(ukey[(size_t)i] & 0xFFFFFFFFu);
        }
        // blocks: load ascending, then block index
        for (int64_t c = 0; c < G; ++c)
          if (load[(size_t)c] >= ((int64_t)1 << 40)) fits = false;
        if (!counting(G, [&](int64_t c) { return load[(size_t)c]; }, false, bord)) {
          for (int64_t c = 0; c < G; ++c)
            bkey[(size_t)c] = ((uint64_t)load[(size_t)c] << 16) | (uint64_t)c;
          std::sort(bkey.begin(), bkey.end());
          for (int64_t c = 0; c < G; ++c) bord[(size_t)c] = (int32_t)(bkey[(size_t)c] & 0xFFFFu);
        }
        for (int64_t i = 0; i < nu; ++i) {
          const int64_t c = bord[(size_t)i];
          const int64_t u = u0 + uord[(size_t)i];
          load[(size_t)c] += cost[(size_t)u];
          order[(size_t)(kk * G + ((kk & 1) ? (G - 1 - c) : c))] = (int32_t)u;
        }
      }
      const double waves = *std::max_element(load.begin(), load.end()) / 4.0;
      if (!(fits && waves < 0.99 * snake)) order.clear();
    }
  }

  p->stats.n_qtiles = (int64_t)p->work.size();
  p->stats.n_tiles = p->stats.n_full + p->stats.n_partial;
  p->stats.n_causal_tiles = causal_tiles;
  p->stats.visible_pairs = visible;

  // ---- workspace layout ----
  size_t off = kStatusBytes;
  p->off_req = off;   off = align_up(off + sizeof(ReqInfo) * B, 256);
  p->off_seg = off;   off = align_up(off + sizeof(int32_t) * (size_t)T, 256);
  p->off_work = off;  off = align_up(off + sizeof(WorkItem) * p->work.size(), 256);
  p->off_klist = off; off = align_up(off + sizeof(uint32_t) * std::max<size_t>(p->klist.size(), 1), 256);
  p->off_order = off; off = align_up(off + sizeof(int32_t) * p->order.size(), 256);
  p->total = off;
  p->stats.workspace_bytes = (int64_t)off;
  return MIS_OK;
}

}  // namespace


}  // namespace mis

namespace mis {

// Cached-prefix plan: the new rows are item sets only; request b's shared set
// Q is rows [cache_start, cache_start + S_b) of the cache. On the virtual row
// axis (cache rows from 0, new rows from qbase) every row of item set a sees
// [s0, pend) = its cached prefix and [lo(j), j] = its own item, which is the
// same two-interval form as a packed request, so the kernel's visibility
// test is unchanged. Cache key tiles never mix with new rows: qbase starts at
// least one 128-row tile past the cache end.
mis_status_t build_plan_cached(const mis_cached_desc* d, HostPlan* p) {
  if (!d || !p) return MIS_ERR_INVALID_ARG;
  if (d->B < 1 || d->T < 1 || d->Hq < 1 || d->Hkv < 1 || d->cache_T < 1) return MIS_ERR_INVALID_ARG;
  if (!d->cu_seqlens || !d->item_ptr || !d->item_offsets || !d->cache_start || !d->cache_len)
    return MIS_ERR_INVALID_ARG;
  if (d->Hq % d->Hkv) return MIS_ERR_SHAPE;
  if (d->D != 64 && d->D != 128) return MIS_ERR_UNSUPPORTED;
  if (!(d->scale >= 0.f) || std::isinf(d->scale)) return MIS_ERR_INVALID_ARG;
  const int32_t B = d->B, T = d->T;
  const int32_t* cu = d->cu_seqlens;
  if (cu[0] != 0 || cu[B] != T) return MIS_ERR_SHAPE;
  for (int b = 0; b < B; ++b)
    if (cu[b + 1] <= cu[b]) return MIS_ERR_SHAPE;
  const int64_t qbase = (int64_t)align_up((size_t)d->cache_T, kBN) + kBN;
  if (qbase + T >= ((int64_t)1 << 31) - kBN) return MIS_ERR_SHAPE;

  p->B = B; p->T = T; p->Hq = d->Hq; p->Hkv = d->Hkv; p->D = d->D;
  p->scale = d->scale > 0.f ? d->scale : 1.0f / std::sqrt((float)d->D);
  p->req.assign(B, ReqInfo{});
  p->seg_start.assign(T, 0);
  p->work.clear(); p->klist.clear(); p->tile_map.clear();
  p->stats = mis_plan_stats{};
  p->cached = true;
  p->cache_T = d->cache_T;
  p->qbase = (int32_t)qbase;
  const int32_t Vb = (int32_t)qbase;

  int64_t visible = 0, causal_tiles = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t S = d->cache_len[b], cs = d->cache_start[b];
    if (S < 1 || cs < 0 || (int64_t)cs + S > d->cache_T) return MIS_ERR_SHAPE;
    const int32_t i0 = d->item_ptr[b], i1 = d->item_ptr[b + 1];
    if (i0 < 0 || i1 <= i0 || (b == 0 && i0 != 0)) return MIS_ERR_SHAPE;
    if (d->item_offsets[i0] != cu[b]) return MIS_ERR_SHAPE;
    for (int32_t i = i0; i < i1; ++i) {
      const int32_t a = d->item_offsets[i];
      const int32_t e = (i + 1 < i1) ? d->item_offsets[i + 1] : cu[b + 1];
      if (a < cu[b] || e <= a || e > cu[b + 1]) return MIS_ERR_SHAPE;
      std::fill(p->seg_start.begin() + a, p->seg_start.begin() + e, Vb + a);
      // row d of the item set sees the S cached rows and d + 1 rows of its set
      const int64_t n = e - a;
      visible += n * S + n * (n + 1) / 2;
    }
    p->req[b] = ReqInfo{cs, Vb + cu[b + 1], cs + S, 0};
  }

  // per-thread scratch: keeps its capacity from plan to plan
  thread_local std::vector<Tmp> tmp;
  tmp.clear();
  for (int b = 0; b < B; ++b) {
    const ReqInfo& R = p->req[b];
    const int32_t S = R.pend - R.s0, base = Vb + cu[b], L = cu[b + 1] - cu[b];
    const int32_t ncache = (S + kBN - 1) / kBN;
    const int32_t nqt = (L + kBM - 1) / kBM;
    for (int32_t t = 0; t < nqt; ++t) {
      const int32_t r0 = base + t * kBM;
      const int32_t r1 = std::min(r0 + kBM, R.e0);
      // a causal pass over [prefix ; items] would need every prefix tile and
      // every new-row tile up to the query tile
      causal_tiles += ncache + (r1 - 1 - base) / kBN + 1;
      const int32_t lo_min = p->seg_start[r0 - Vb], lo_max = p->seg_start[r1 - 1 - Vb];
      Tmp w{b, r0, (int32_t)p->klist.size(), 0, 0, 0, 0, (int64_t)tmp.size()};
      auto emit = [&](int32_t u, int32_t c0, bool full, bool need_mask) {
        p->klist.push_back((uint32_t)c0 | (need_mask ? kNeedMask : 0u));
        p->tile_map.insert(p->tile_map.end(), {b, t, u, full ? 1 : 2});
        if (full) ++p->stats.n_full; else ++p->stats.n_partial;
        const int c = need_mask ? 5 : 4;
        (w.nk % 2 ? w.cost_odd : w.cost_even) += c;
        ++w.nk;
        w.cost += c;
      };
      // the cached prefix: every row sees all of it; a tile that runs past the
      // prefix end holds other rows of the cache and is masked there
      for (int32_t u = 0; u < ncache; ++u) {
        const int32_t c0 = R.s0 + u * kBN;
        emit(u, c0, true, c0 + kBN > R.pend);
      }
      // the band of the query tile's own items
      const int32_t ba = (lo_min - base) / kBN, bb = (r1 - 1 - base) / kBN + 1;
      for (int32_t v = ba; v < bb; ++v) {
        const int32_t c0 = base + v * kBN;
        const int32_t c1 = std::min(c0 + kBN, R.e0);
        const bool full = (c1 - 1 <= r0) && (c0 >= lo_max);
        emit(ncache + v, c0, full, !full || c0 + kBN > R.e0);
      }
      tmp.push_back(w);
    }
  }
  return finish_plan(p, tmp, B, T, visible, causal_tiles);
}

}  // namespace mis

// ---------------------------------------------------------------------------
// Layout packing (C ABI). Rows of request b: P_b prefix tokens, the leading
// DELIM, then for each item its L_i tokens and a trailing DELIM
// ("Turbocharging ...", section "Multi-item-scoring: Our innovation with
// SGLang"). Position ids follow Section 4.1 of "From Generation to Scoring":
// the shared rows get 0..S_b-1 and offset d of every item set gets S_b + d.
// ---------------------------------------------------------------------------
extern "C" mis_status_t mis_layout_size(int32_t B, const int32_t* prefix_tokens,
                                        const int32_t* n_items, const int32_t* item_lens,
                                        int64_t* T_out, int64_t* M_out) {
  if (B < 1 || !prefix_tokens || !n_items) return MIS_ERR_INVALID_ARG;
  int64_t T = 0, M = 0;
  for (int32_t b = 0; b < B; ++b) {
    if (prefix_tokens[b] < 0 || n_items[b] < 0) return MIS_ERR_INVALID_ARG;
    T += (int64_t)prefix_tokens[b] + 1;
    M += n_items[b];
  }
  if (M > 0 && !item_lens) return MIS_ERR_INVALID_ARG;
  for (int64_t i = 0; i < M; ++i) {
    if (item_lens[i] < 0) return MIS_ERR_INVALID_ARG;
    T += (int64_t)item_lens[i] + 1;
  }
  if (T >= ((int64_t)1 << 31) - mis::kBN) return MIS_ERR_SHAPE;
  if (T_out) *T_out = T;
  if (M_out) *M_out = M;
  return MIS_OK;
}

extern "C" mis_status_t mis_build_layout(int32_t B, const int32_t* prefix_tokens,
                                         const int32_t* n_items, const int32_t* item_lens,
                                         int32_t* cu_seqlens, int32_t* prefix_len,
                                         int32_t* item_ptr, int32_t* item_offsets,
                                         int32_t* delim_positions, int32_t* position_ids,
                                         int64_t position_cap) {
  int64_t T = 0, M = 0;
  mis_status_t st = mis_layout_size(B, prefix_tokens, n_items, item_lens, &T, &M);
  if (st != MIS_OK) return st;
  if (!cu_seqlens || !prefix_len || !item_ptr) return MIS_ERR_INVALID_ARG;
  if (M > 0 && (!item_offsets || !delim_positions)) return MIS_ERR_INVALID_ARG;
  if (position_ids && position_cap < T) return MIS_ERR_SHAPE;
  int32_t row = 0, it = 0;
  cu_seqlens[0] = 0;
  item_ptr[0] = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t S = prefix_tokens[b] + 1;
    prefix_len[b] = S;
    if (position_ids)
      for (int32_t t = 0; t < S; ++t) position_ids[row + t] = t;
    row += S;
    for (int32_t n = 0; n < n_items[b]; ++n, ++it) {
      const int32_t len = item_lens[it] + 1;     // item tokens + trailing DELIM
      item_offsets[it] = row;
      if (position_ids)
        for (int32_t t = 0; t < len; ++t) position_ids[row + t] = S + t;
      row += len;
      delim_positions[it] = row - 1;
    }
    cu_seqlens[b + 1] = row;
    item_ptr[b + 1] = it;
  }
  return MIS_OK;
}

// ---------------------------------------------------------------------------
// Setwise layout (C ABI): per request its query tokens, every candidate's
// tokens, then one marker per candidate, as one plain causal sequence; the
// marker rows are the readout rows, in candidate order ("Scaling JEV-like
// Decision Models with SGLang", "Benchmark: Fused-Choice vs. Setwise Scoring").
// ---------------------------------------------------------------------------
extern "C" mis_status_t mis_setwise_layout_size(int32_t B, const int32_t* query_tokens,
                                                const int32_t* n_cands, const int32_t* cand_lens,
                                                int64_t* T_out, int64_t* M_out) {
  if (B < 1 || !query_tokens || !n_cands) return MIS_ERR_INVALID_ARG;
  int64_t T = 0, M = 0;
  for (int32_t b = 0; b < B; ++b) {
    if (query_tokens[b] < 0 || n_cands[b] < 0) return MIS_ERR_INVALID_ARG;
    if (query_tokens[b] == 0 && n_cands[b] == 0) return MIS_ERR_SHAPE;   // empty request
    T += (int64_t)query_tokens[b] + n_cands[b];                           // query + markers
    M += n_cands[b];
  }
  if (M > 0 && !cand_lens) return MIS_ERR_INVALID_ARG;
  for (int64_t i = 0; i < M; ++i) {
    if (cand_lens[i] < 0) return MIS_ERR_INVALID_ARG;
    T += cand_lens[i];
  }
  if (T >= ((int64_t)1 << 31) - mis::kBN) return MIS_ERR_SHAPE;
  if (T_out) *T_out = T;
  if (M_out) *M_out = M;
  return MIS_OK;
}

extern "C" mis_status_t mis_build_setwise_layout(int32_t B, const int32_t* query_tokens,
                                                 const int32_t* n_cands, const int32_t* cand_lens,
                                                 int32_t* cu_seqlens, int32_t* prefix_len,
                                                 int32_t* marker_positions, int32_t* position_ids,
                                                 int64_t position_cap) {
  int64_t T = 0, M = 0;
  mis_status_t st = mis_setwise_layout_size(B, query_tokens, n_cands, cand_lens, &T, &M);
  if (st != MIS_OK) return st;
  if (!cu_seqlens || !prefix_len) return MIS_ERR_INVALID_ARG;
  if (M > 0 && !marker_positions) return MIS_ERR_INVALID_ARG;
  if (position_ids && position_cap < T) return MIS_ERR_SHAPE;
  int32_t row = 0, c = 0, m = 0;
  cu_seqlens[0] = 0;
  for (int32_t b = 0; b < B; ++b) {
    int32_t len = query_tokens[b];
    for (int32_t i = 0; i < n_cands[b]; ++i) len += cand_lens[c + i];
    c += n_cands[b];
    for (int32_t i = 0; i < n_cands[b]; ++i) marker_positions[m++] = row + len + i;
    len += n_cands[b];
    if (position_ids)
      for (int32_t t = 0; t < len; ++t) position_ids[row + t] = t;
    prefix_len[b] = len;                 // every row in the shared set: plain causal
    row += len;
    cu_seqlens[b + 1] = row;
  }
  return MIS_OK;
}
