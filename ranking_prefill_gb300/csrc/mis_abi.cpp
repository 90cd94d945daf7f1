// C ABI of the MIS library: argument checks, plan lifecycle, tensor maps,
// device status. No C++ exception crosses this boundary.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "mis_internal.h"

namespace mis {

namespace {

std::atomic<uint64_t> g_wait_limit_ns{200ull * 1000 * 1000};
std::atomic<uint32_t> g_inject_stall{0};
std::atomic<int32_t> g_schedule{MIS_SCHEDULE_AUTO};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }
uint32_t inject_stall_mask() { return g_inject_stall.load(); }
int32_t schedule_override() { return g_schedule.load(); }

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

namespace {

// A few recently encoded tensor maps (the LM head, a layer's Q/K/V buffers
// are reused call after call); encoding is pure host work, so a hit only
// saves time and a miss re-encodes.
struct TmapKey {
  const void* base;
  int rank;
  uint64_t dims[3], strides[2];
  uint32_t box[3];
  bool operator==(const TmapKey& o) const {
    return base == o.base && rank == o.rank && std::memcmp(dims, o.dims, sizeof(dims)) == 0 &&
           std::memcmp(strides, o.strides, sizeof(strides)) == 0 &&
           std::memcmp(box, o.box, sizeof(box)) == 0;
  }
};
constexpr int kTmapCache = 16;
std::mutex g_tmap_mu;
TmapKey g_tmap_key[kTmapCache];
CUtensorMap g_tmap_val[kTmapCache];
int g_tmap_n = 0, g_tmap_next = 0;

}  // namespace

// bf16 tiled tensor map with 128-byte swizzle; dims/box innermost first.
CUtensorMap make_tmap_bf16(const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box, bool* ok) {
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  TmapKey key;
  std::memset(&key, 0, sizeof(key));
  key.base = base;
  key.rank = rank;
  for (int i = 0; i < rank && i < 3; ++i) { key.dims[i] = dims[i]; key.box[i] = box[i]; }
  for (int i = 0; i + 1 < rank && i < 2; ++i) key.strides[i] = strides_bytes[i];
  {
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    for (int i = 0; i < g_tmap_n; ++i)
      if (g_tmap_key[i] == key) return g_tmap_val[i];
  }
  auto fn = encode_fn();
  if (!fn) { *ok = false; return m; }
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) { gd[i] = dims[i]; bx[i] = box[i]; es[i] = 1; }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base),
                  gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *ok = false;
    return m;
  }
  std::lock_guard<std::mutex> lock(g_tmap_mu);
  g_tmap_key[g_tmap_next] = key;
  g_tmap_val[g_tmap_next] = m;
  g_tmap_next = (g_tmap_next + 1) % kTmapCache;
  if (g_tmap_n < kTmapCache) ++g_tmap_n;
  return m;
}

bool kernel_attr_once(const void* kernel, int smem_bytes) {
  // cudaFuncSetAttribute is per device; remember which (kernel, device) pairs
  // are done
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& d : done)
    if (d.first == kernel && d.second == dev) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
      cudaSuccess)
    return false;
  done.emplace_back(kernel, dev);
  return true;
}

}  // namespace mis

struct mis_plan_s {
  mis::HostPlan p;
};

const mis::HostPlan& mis::plan_of(mis_plan_t plan) { return plan->p; }

namespace {

// Destroyed plans are kept (a few) and handed out again: a serving loop that
// plans every batch then reuses the same host buffers instead of faulting in
// fresh pages for every plan.
constexpr size_t kPlanPoolMax = 4;
std::mutex g_plan_pool_mu;
std::vector<mis_plan_s*> g_plan_pool;

mis_plan_s* new_plan() {
  {
    std::lock_guard<std::mutex> lock(g_plan_pool_mu);
    if (!g_plan_pool.empty()) {
      mis_plan_s* h = g_plan_pool.back();
      g_plan_pool.pop_back();
      h->p.reset();
      return h;
    }
  }
  return new mis_plan_s();
}

void free_plan(mis_plan_s* h) {
  if (!h) return;
  {
    std::lock_guard<std::mutex> lock(g_plan_pool_mu);
    if (g_plan_pool.size() < kPlanPoolMax) {
      g_plan_pool.push_back(h);
      return;
    }
  }
  free_plan(h);
}

}  // namespace

using namespace mis;

extern "C" {

const char* mis_status_string(int status) {
  switch (status) {
    case MIS_OK: return "ok";
    case MIS_ERR_INVALID_ARG: return "invalid argument";
    case MIS_ERR_SHAPE: return "inconsistent shape, offsets or strides";
    case MIS_ERR_UNSUPPORTED: return "unsupported configuration";
    case MIS_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MIS_ERR_CUDA: return "CUDA call failed";
    case MIS_ERR_DEVICE_TIMEOUT: return "a device wait ran out of time";
    case MIS_ERR_DEVICE_INDEX: return "a device-side index was out of range";
    default: return "unknown status";
  }
}

int mis_abi_version(void) { return MIS_ABI_VERSION; }

uint64_t mis_set_wait_limit_ns(uint64_t ns) { return g_wait_limit_ns.exchange(ns); }

uint32_t mis_inject_stall(uint32_t mask) { return g_inject_stall.exchange(mask); }

int32_t mis_set_schedule(int32_t mode) {
  if (mode != MIS_SCHEDULE_AUTO && mode != MIS_SCHEDULE_PAIR && mode != MIS_SCHEDULE_SPLIT)
    return -1;
  return g_schedule.exchange(mode);
}

size_t mis_plan_workspace_size(const mis_attn_desc* desc) {
  try {
    HostPlan p;
    if (build_plan(desc, &p) != MIS_OK) return 0;
    return p.total;
  } catch (...) {
    return 0;
  }
}

}  // extern "C"

namespace {

// Build a plan with `build` and upload it into `workspace` (or keep it
// host-only when workspace is NULL and ws_bytes is 0).
template <typename Desc, typename Build>
mis_status_t create_plan(const Desc* desc, Build build, void* workspace, size_t ws_bytes,
                         void* stream, mis_plan_t* out) {
  if (!out) return MIS_ERR_INVALID_ARG;
  *out = nullptr;
  mis_plan_s* h = nullptr;
  try {
    h = new_plan();
    mis_status_t st = build(desc, &h->p);
    if (st != MIS_OK) { free_plan(h); return st; }
    HostPlan& p = h->p;
    if (!workspace && ws_bytes == 0) {   // host-only plan: inspection, no launches
      *out = h;
      return MIS_OK;
    }
    if (!workspace || !aligned256(workspace) || ws_bytes < p.total) { free_plan(h); return MIS_ERR_WORKSPACE; }
    p.workspace = workspace;
    // one host image of the workspace after the status words, one copy
    std::vector<uint8_t> img(p.total - kStatusBytes, 0);
    auto put = [&](size_t off, const void* src, size_t n) {
      if (n) std::memcpy(img.data() + (off - kStatusBytes), src, n);
    };
    put(p.off_req, p.req.data(), p.req.size() * sizeof(ReqInfo));
    put(p.off_seg, p.seg_start.data(), p.seg_start.size() * sizeof(int32_t));
    put(p.off_work, p.work.data(), p.work.size() * sizeof(WorkItem));
    put(p.off_klist, p.klist.data(), p.klist.size() * sizeof(uint32_t));
    put(p.off_order, p.order.data(), p.order.size() * sizeof(int32_t));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    if (cudaMemsetAsync(ws, 0, kStatusBytes, s) != cudaSuccess ||
        cudaMemcpyAsync(ws + kStatusBytes, img.data(), img.size(), cudaMemcpyHostToDevice, s) !=
            cudaSuccess) {
      free_plan(h);
      return MIS_ERR_CUDA;
    }
    // A copy from pageable memory returns once the source has been staged, so
    // `img` may be released when this function returns.
    *out = h;
    return MIS_OK;
  } catch (...) {
    free_plan(h);
    return MIS_ERR_INVALID_ARG;
  }
}

}  // namespace

extern "C" {

mis_status_t mis_plan_create(const mis_attn_desc* desc, void* workspace, size_t ws_bytes,
                             void* stream, mis_plan_t* out) {
  return create_plan(desc, build_plan, workspace, ws_bytes, stream, out);
}

size_t mis_cached_plan_workspace_size(const mis_cached_desc* desc) {
  try {
    HostPlan p;
    if (build_plan_cached(desc, &p) != MIS_OK) return 0;
    return p.total;
  } catch (...) {
    return 0;
  }
}

mis_status_t mis_cached_plan_create(const mis_cached_desc* desc, void* workspace, size_t ws_bytes,
                                    void* stream, mis_plan_t* out) {
  return create_plan(desc, build_plan_cached, workspace, ws_bytes, stream, out);
}

}  // extern "C"

struct mis_planner_s {
  void* staging[2] = {nullptr, nullptr};
  size_t cap[2] = {0, 0};
  cudaEvent_t done[2] = {nullptr, nullptr};
  bool used[2] = {false, false};
  int next = 0;
};

extern "C" {

mis_status_t mis_planner_create(mis_planner_t* out) {
  if (!out) return MIS_ERR_INVALID_ARG;
  *out = nullptr;
  mis_planner_s* pl = nullptr;
  try {
    pl = new mis_planner_s();
  } catch (...) {
    return MIS_ERR_INVALID_ARG;
  }
  for (int i = 0; i < 2; ++i)
    if (cudaEventCreateWithFlags(&pl->done[i], cudaEventDisableTiming) != cudaSuccess) {
      mis_planner_destroy(pl);
      return MIS_ERR_CUDA;
    }
  *out = pl;
  return MIS_OK;
}

mis_status_t mis_planner_destroy(mis_planner_t pl) {
  if (!pl) return MIS_OK;
  for (int i = 0; i < 2; ++i) {
    if (pl->done[i]) {
      if (pl->used[i]) cudaEventSynchronize(pl->done[i]);
      cudaEventDestroy(pl->done[i]);
    }
    if (pl->staging[i]) cudaFreeHost(pl->staging[i]);
  }
  delete pl;
  return MIS_OK;
}

mis_status_t mis_planner_plan(mis_planner_t pl, const mis_attn_desc* desc, void* workspace,
                              size_t ws_bytes, const void* extra_host, size_t extra_bytes,
                              void* stream, mis_plan_t* out) {
  if (!pl || !out || (extra_bytes && !extra_host)) return MIS_ERR_INVALID_ARG;
  *out = nullptr;
  mis_plan_s* h = nullptr;
  try {
    h = new_plan();
    mis_status_t st = build_plan(desc, &h->p);
    if (st != MIS_OK) { free_plan(h); return st; }
    HostPlan& p = h->p;
    if (!workspace || !aligned256(workspace) || ws_bytes < p.total + extra_bytes) {
      free_plan(h);
      return MIS_ERR_WORKSPACE;
    }
    p.workspace = workspace;
    const int b = pl->next;
    // one image from offset 0: zeroed status words, the plan, the side payload
    const size_t n = p.total + extra_bytes;
    // the buffer's previous upload (two calls ago) must have been read
    if (pl->used[b] && cudaEventSynchronize(pl->done[b]) != cudaSuccess) { free_plan(h); return MIS_ERR_CUDA; }
    if (pl->cap[b] < n) {
      if (pl->staging[b]) cudaFreeHost(pl->staging[b]);
      pl->staging[b] = nullptr;
      pl->cap[b] = 0;
      const size_t want = n + n / 2 + 4096;
      if (cudaHostAlloc(&pl->staging[b], want, cudaHostAllocDefault) != cudaSuccess) {
        pl->staging[b] = nullptr;
        free_plan(h);
        return MIS_ERR_CUDA;
      }
      pl->cap[b] = want;
    }
    uint8_t* img = static_cast<uint8_t*>(pl->staging[b]);
    std::memset(img, 0, kStatusBytes);   // the status words; every region is written below
    auto put = [&](size_t off, const void* src, size_t len) {
      if (len) std::memcpy(img + off, src, len);
    };
    put(p.off_req, p.req.data(), p.req.size() * sizeof(ReqInfo));
    put(p.off_seg, p.seg_start.data(), p.seg_start.size() * sizeof(int32_t));
    put(p.off_work, p.work.data(), p.work.size() * sizeof(WorkItem));
    put(p.off_klist, p.klist.data(), p.klist.size() * sizeof(uint32_t));
    put(p.off_order, p.order.data(), p.order.size() * sizeof(int32_t));
    put(p.total, extra_host, extra_bytes);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(workspace, img, n, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaEventRecord(pl->done[b], s) != cudaSuccess) {
      free_plan(h);
      return MIS_ERR_CUDA;
    }
    p.status_clear = true;
    pl->used[b] = true;
    pl->next = b ^ 1;
    *out = h;
    return MIS_OK;
  } catch (...) {
    free_plan(h);
    return MIS_ERR_INVALID_ARG;
  }
}

mis_status_t mis_plan_get_stats(mis_plan_t plan, mis_plan_stats* out) {
  if (!plan || !out) return MIS_ERR_INVALID_ARG;
  *out = plan->p.stats;
  return MIS_OK;
}

mis_status_t mis_plan_tile_map(mis_plan_t plan, int32_t* host_out, size_t cap, size_t* n_out) {
  if (!plan || !n_out || (cap && !host_out)) return MIS_ERR_INVALID_ARG;
  const std::vector<int32_t>& tm = plan->p.tile_map;
  const size_t n = tm.size() / 4;
  *n_out = n;
  const size_t w = cap < n ? cap : n;
  if (w) std::memcpy(host_out, tm.data(), w * 4 * sizeof(int32_t));
  return MIS_OK;
}

mis_status_t mis_plan_unit_walk(mis_plan_t plan, int32_t* host_out, size_t cap, size_t* n_out,
                                int32_t* blocks_out) {
  if (!plan || !n_out || (cap && !host_out)) return MIS_ERR_INVALID_ARG;
  const HostPlan& p = plan->p;
  const int64_t units = p.stats.n_units;
  const size_t n = p.order.empty() ? (size_t)units : p.order.size();
  *n_out = n;
  if (blocks_out) *blocks_out = (int32_t)std::min<int64_t>(units, num_sms());
  const size_t w = cap < n ? cap : n;
  for (size_t i = 0; i < w; ++i) host_out[i] = p.order.empty() ? (int32_t)i : p.order[i];
  return MIS_OK;
}

mis_status_t mis_plan_exec_tiles(mis_plan_t plan, int32_t* host_out, size_t cap, size_t* n_out) {
  if (!plan || !n_out || (cap && !host_out)) return MIS_ERR_INVALID_ARG;
  const HostPlan& p = plan->p;
  size_t n = 0;
  for (const WorkItem& w : p.work) {
    for (int32_t i = 0; i < w.nk; ++i, ++n) {
      if (n >= cap) continue;
      const uint32_t e = p.klist[(size_t)w.kofs + i];
      int32_t* q = host_out + 4 * n;
      q[0] = w.req;
      q[1] = w.q0;
      q[2] = (int32_t)(e & ~kNeedMask);
      q[3] = (e & kNeedMask) ? 1 : 0;
    }
  }
  *n_out = n;
  return MIS_OK;
}

mis_status_t mis_plan_destroy(mis_plan_t plan) {
  free_plan(plan);
  return MIS_OK;
}

mis_status_t mis_attention_fwd_plan(mis_plan_t plan, const void* q, const void* k, const void* v,
                                    void* o, float* lse, int64_t qs, int64_t ks, int64_t vs,
                                    int64_t os, void* stream) {
  if (!plan) return MIS_ERR_INVALID_ARG;
  HostPlan& p = plan->p;
  if (p.cached) return MIS_ERR_INVALID_ARG;       // needs the cache buffers
  if (!p.workspace) return MIS_ERR_WORKSPACE;
  if (!q || !k || !v || !o) return MIS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return MIS_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return MIS_ERR_INVALID_ARG;
  const int64_t wq = (int64_t)p.Hq * p.D, wk = (int64_t)p.Hkv * p.D;
  if (qs < wq || os < wq || ks < wk || vs < wk) return MIS_ERR_SHAPE;
  if ((qs | ks | vs | os) & 7) return MIS_ERR_SHAPE;
  try {
    return launch_attention(p, q, k, v, nullptr, nullptr, o, lse, qs, ks, vs, 0, 0, os, stream);
  } catch (...) {
    return MIS_ERR_CUDA;
  }
}

mis_status_t mis_attention_fwd_plan_rope(mis_plan_t plan, const void* q, const void* k,
                                         const void* v, void* o, float* lse, int64_t qs,
                                         int64_t ks, int64_t vs, int64_t os, double rope_base,
                                         void* stream) {
  if (!plan) return MIS_ERR_INVALID_ARG;
  HostPlan& p = plan->p;
  if (p.cached) return MIS_ERR_INVALID_ARG;       // needs the cache buffers
  if (!p.workspace) return MIS_ERR_WORKSPACE;
  if (!q || !k || !v || !o) return MIS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return MIS_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return MIS_ERR_INVALID_ARG;
  if (!(rope_base > 1.0) || !std::isfinite(rope_base)) return MIS_ERR_INVALID_ARG;
  // positions stay below the longest request's length, at most 2^17: the
  // range reduction of the fp32 angle p * base^(-2i/D) is then exact
  int64_t longest = 0;
  for (const ReqInfo& r : p.req) longest = std::max<int64_t>(longest, r.e0 - r.s0);
  if (longest > (1 << 17)) return MIS_ERR_UNSUPPORTED;
  const int64_t wq = (int64_t)p.Hq * p.D, wk = (int64_t)p.Hkv * p.D;
  if (qs < wq || os < wq || ks < wk || vs < wk) return MIS_ERR_SHAPE;
  if ((qs | ks | vs | os) & 7) return MIS_ERR_SHAPE;
  const RopeQ rope{rope_base};
  try {
    return launch_attention(p, q, k, v, nullptr, nullptr, o, lse, qs, ks, vs, 0, 0, os, stream,
                            &rope);
  } catch (...) {
    return MIS_ERR_CUDA;
  }
}

mis_status_t mis_attention_fwd_cached(mis_plan_t plan, const void* q, const void* k,
                                      const void* v, const void* k_cache, const void* v_cache,
                                      void* o, float* lse, int64_t qs, int64_t ks, int64_t vs,
                                      int64_t kcs, int64_t vcs, int64_t os, void* stream) {
  if (!plan) return MIS_ERR_INVALID_ARG;
  HostPlan& p = plan->p;
  if (!p.cached) return MIS_ERR_INVALID_ARG;
  if (!p.workspace) return MIS_ERR_WORKSPACE;
  if (!q || !k || !v || !o || !k_cache || !v_cache) return MIS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(k_cache) ||
      !aligned16(v_cache))
    return MIS_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return MIS_ERR_INVALID_ARG;
  const int64_t wq = (int64_t)p.Hq * p.D, wk = (int64_t)p.Hkv * p.D;
  if (qs < wq || os < wq || ks < wk || vs < wk || kcs < wk || vcs < wk) return MIS_ERR_SHAPE;
  if ((qs | ks | vs | kcs | vcs | os) & 7) return MIS_ERR_SHAPE;
  try {
    return launch_attention(p, q, k, v, k_cache, v_cache, o, lse, qs, ks, vs, kcs, vcs, os, stream);
  } catch (...) {
    return MIS_ERR_CUDA;
  }
}

mis_status_t mis_attention_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                               int64_t qs, int64_t ks, int64_t vs, int64_t os,
                               const mis_attn_desc* desc, void* workspace, size_t ws_bytes,
                               void* stream) {
  mis_plan_t plan = nullptr;
  mis_status_t st = mis_plan_create(desc, workspace, ws_bytes, stream, &plan);
  if (st != MIS_OK) return st;
  st = mis_attention_fwd_plan(plan, q, k, v, o, lse, qs, ks, vs, os, stream);
  mis_plan_destroy(plan);
  return st;
}

size_t mis_label_scores_workspace_size(int32_t M, int32_t d, int32_t V, int32_t K) {
  if (M < 0 || d <= 0 || V <= 0 || K <= 0) return 0;
  return score_workspace_size(M, d, V, K);
}

mis_status_t mis_label_scores(const void* hidden, int64_t hidden_row_stride, int32_t T,
                              const void* w_lm, int32_t d, int32_t V,
                              const int32_t* delim_positions, int32_t M,
                              const int32_t* label_token_ids, int32_t K, float* out_logprobs,
                              float* out_renorm, void* workspace, size_t ws_bytes, void* stream) {
  if (M < 0 || T < 1 || V < 1 || d < 1 || K < 1) return MIS_ERR_INVALID_ARG;
  if (K > 16) return MIS_ERR_UNSUPPORTED;
  if (d % 64 || d > 8192) return MIS_ERR_UNSUPPORTED;
  if (!label_token_ids) return MIS_ERR_INVALID_ARG;
  for (int l = 0; l < K; ++l)
    if (label_token_ids[l] < 0 || label_token_ids[l] >= V) return MIS_ERR_INVALID_ARG;
  if (M > 0) {
    if (!hidden || !w_lm || !delim_positions || !out_logprobs) return MIS_ERR_INVALID_ARG;
    if (!aligned16(hidden) || !aligned16(w_lm)) return MIS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(delim_positions) | reinterpret_cast<uintptr_t>(out_logprobs) |
         reinterpret_cast<uintptr_t>(out_renorm)) & 3u)
      return MIS_ERR_INVALID_ARG;
    if (hidden_row_stride < d || (hidden_row_stride & 7)) return MIS_ERR_SHAPE;
  }
  if (!workspace || !aligned256(workspace)) return MIS_ERR_WORKSPACE;
  if (ws_bytes < score_workspace_size(M, d, V, K)) return MIS_ERR_WORKSPACE;
  ScoreArgs a;
  a.hidden = hidden; a.hidden_stride = hidden_row_stride; a.T = T;
  a.w_lm = w_lm; a.d = d; a.V = V;
  a.delim = delim_positions; a.M = M;
  for (int l = 0; l < 16; ++l) a.labels[l] = l < K ? label_token_ids[l] : -1;
  a.K = K;
  a.out_logprobs = out_logprobs; a.out_renorm = out_renorm;
  a.workspace = workspace; a.ws_bytes = ws_bytes;
  try {
    return launch_score(a, stream);
  } catch (...) {
    return MIS_ERR_CUDA;
  }
}

mis_status_t mis_get_device_status(const void* workspace, void* stream) {
  if (!workspace) return MIS_ERR_INVALID_ARG;
  uint32_t w[2] = {0, 0};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(w, workspace, sizeof(w), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MIS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MIS_ERR_CUDA;
  if (w[0] & kDevTimeout) return MIS_ERR_DEVICE_TIMEOUT;
  if (w[0] & kDevIndex) return MIS_ERR_DEVICE_INDEX;
  return MIS_OK;
}

}  // extern "C"
