// Internal declarations shared by the host-side translation units of the
// MIS library. Nothing here is part of the C ABI (include/mis.h is).
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/mis.h"

namespace mis {

// Attention tiling: 128 query rows x 128 keys per block.
constexpr int kBM = 128;
constexpr int kBN = 128;

// Workspace layout: the first 256 bytes hold the device status words.
constexpr size_t kStatusBytes = 256;
// Bits of the device status word (workspace offset 0).
constexpr uint32_t kDevTimeout = 1u;
constexpr uint32_t kDevIndex = 2u;

// Key-tile list entry: absolute first key row | (needs element mask << 31).
constexpr uint32_t kNeedMask = 0x80000000u;

struct ReqInfo {   // one request of the packed batch, absolute rows
  int32_t s0;      // first row
  int32_t e0;      // one past the last row
  int32_t pend;    // s0 + S_b: rows [s0, pend) form the shared set Q
  int32_t pad;
};

struct WorkItem {  // one (request, 128-row query tile)
  int32_t req;
  int32_t q0;      // absolute first query row
  int32_t kofs;    // first entry in the key-tile list
  int32_t nk;      // number of key tiles
};

struct HostPlan {
  int32_t B = 0, T = 0, Hq = 0, Hkv = 0, D = 0;
  float scale = 0.f;
  std::vector<ReqInfo> req;
  std::vector<int32_t> seg_start;  // [T] first row of the set (Q or I_i) holding each row
  std::vector<WorkItem> work;      // heaviest first
  std::vector<uint32_t> klist;
  std::vector<int32_t> tile_map;   // canonical quadruples
  mis_plan_stats stats{};
  // byte offsets inside the device workspace
  size_t off_req = 0, off_seg = 0, off_work = 0, off_klist = 0, total = 0;
  bool split = false;              // split schedule (one head per unit, key tiles alternate
                                   // between the block's two softmax streams)
  int32_t n_head_groups = 1;       // units per query tile: Hq / 2 (pair) or Hq (split)
  // the unit at each walk position of the kernel's blocks (pass kk, block c
  // at kk * G + c, odd passes reversed), -1 for none; empty: position = unit
  std::vector<int32_t> order;
  size_t off_order = 0;
  void* workspace = nullptr;       // device base, set by mis_plan_create
  bool status_clear = false;       // the upload zeroed the status words; the
                                   // first launch need not clear them again
  // cached-prefix plans: keys of request b's shared set live in a separate
  // cache buffer. Rows are numbered on one virtual axis: cache rows
  // [0, cache_T), new rows from qbase on (qbase leaves at least one empty
  // 128-row tile after the cache, so no cache key tile reaches a new row).
  bool cached = false;
  int32_t cache_T = 0;
  int32_t qbase = 0;

  // Back to the state of a fresh plan; the vectors keep their capacity, so a
  // recycled plan of similar size touches no fresh pages.
  void reset() {
    B = T = Hq = Hkv = D = 0;
    scale = 0.f;
    req.clear(); seg_start.clear(); work.clear(); klist.clear(); tile_map.clear(); order.clear();
    stats = mis_plan_stats{};
    off_req = off_seg = off_work = off_klist = off_order = total = 0;
    split = false;
    n_head_groups = 1;
    workspace = nullptr;
    status_clear = false;
    cached = false;
    cache_T = 0;
    qbase = 0;
  }
};

// The host plan behind a C-ABI plan handle.
const HostPlan& plan_of(mis_plan_t plan);

// Validates a cached-prefix descriptor and fills the plan (cached = true).
mis_status_t build_plan_cached(const mis_cached_desc* d, HostPlan* p);

// Validates the descriptor and fills everything but `workspace`.
mis_status_t build_plan(const mis_attn_desc* d, HostPlan* p);

// Per-device properties the launchers need (cached).
int num_sms();

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel in the stream drains; every kernel of this library calls
// griddepcontrol.wait before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Raise a kernel's dynamic shared-memory limit once per device.
bool kernel_attr_once(const void* kernel, int smem_bytes);

// Process-wide wait limit for the kernels' bounded waits.
uint64_t wait_limit_ns();
// Process-wide failure-injection mask (bit 0: attention, bit 1: scoring).
uint32_t inject_stall_mask();
// Process-wide attention schedule override (MIS_SCHEDULE_*).
int32_t schedule_override();

// Rotary embedding of Q on load at the reused position ids (the base of the
// rotate-half frequencies base^(-2i/D)).
struct RopeQ {
  double base;
};

// Kernel launchers (defined in the .cu files). Return MIS_ERR_CUDA on launch
// failure. Pointers are already validated.
// k_cache / v_cache (and their strides) are used by cached plans only; rope
// (or null) rotates Q on load.
mis_status_t launch_attention(HostPlan& p, const void* q, const void* k, const void* v,
                              const void* k_cache, const void* v_cache, void* o, float* lse,
                              int64_t qs, int64_t ks, int64_t vs, int64_t kcs, int64_t vcs,
                              int64_t os, void* stream, const RopeQ* rope = nullptr);

struct ScoreArgs {
  const void* hidden; int64_t hidden_stride; int32_t T;
  const void* w_lm; int32_t d; int32_t V;
  const int32_t* delim; int32_t M;
  int32_t labels[16]; int32_t K;
  float* out_logprobs; float* out_renorm;
  void* workspace; size_t ws_bytes;
};
size_t score_workspace_size(int32_t M, int32_t d, int32_t V, int32_t K);
mis_status_t launch_score(const ScoreArgs& a, void* stream);

}  // namespace mis
