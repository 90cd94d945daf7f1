// Rotary position embedding of Q and K at given position ids, sm_103a.
//
// The position ids are the reused ones of "From Generation to Scoring",
// Section 4.1 (query 0..S-1, offset d of every item set -> S + d), so each
// item's rows are rotated exactly as in its own single-item prompt
// ("Turbocharging LinkedIn's recommendation systems with SGLang", "SGLang
// changes": positional encoding adjusted so each item aligns with its
// single-item position). Rotate-half form: for i < D/2 the pair
// (x[i], x[i + D/2]) of a row at position p turns by p * base^(-2i/D).
//
// HBM-bound: every element of Q and K is read and written once. One thread
// owns one row's 8-pair chunk for a group of heads of that row (Q heads
// first, then K heads), so the 8 angles' sines and cosines serve the whole
// group. A row's heads are split over several threads only for short batches,
// whose (row, chunk) cells alone would fill less than half of about 2,048
// threads per SM; long batches compute each angle once per row. Consecutive
// threads cover consecutive 16-byte chunks of a row (coalesced). The inverse frequencies arrive precomputed in fp64 and rounded
// to fp32, so the only float32 error in an angle is the rounding of p * f.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "mis_internal.h"
#include "mis_ptx.cuh"

namespace mis {
namespace {

using namespace dev;

constexpr int kRopeThreads = 256;
constexpr int64_t kThreadsPerSm = 2048;

struct RopeParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k;
  __nv_bfloat16* qo;
  __nv_bfloat16* ko;
  int64_t qs, ks, qos, kos;   // row strides, elements
  const int32_t* pos;         // [T] device
  int32_t T, Hq, Hkv;
  int32_t hpt;                // heads per thread
  float inv_freq[64];         // base^(-2i/D), i < D/2
};

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int D>
__global__ void __launch_bounds__(kRopeThreads)
mis_rope_kernel(const RopeParams p) {
  // No early launch of the next kernel: the attention grid that follows is
  // persistent (one block per SM holding the whole register file), and
  // blocks of it arriving early took SMs from this pass's later blocks
  // (measured: decision-256 step 1.61 -> 1.23 ms with the K pass below).
  griddep_wait();
  constexpr int HALF = D / 2, NC = HALF / 8;          // 8-pair chunks per head
  const int H = p.Hq + p.Hkv;
  const int NG = (H + p.hpt - 1) / p.hpt;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int c = (int)(gid % NC);
  const int64_t tg = gid / NC;
  const int grp = (int)(tg % NG);
  const int64_t t = tg / NG;
  if (t >= p.T) return;
  const float fp = (float)p.pos[t];
  float cs[8], sn[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) sincosf(fp * p.inv_freq[c * 8 + e], &sn[e], &cs[e]);

  auto rotate = [&](const __nv_bfloat16* src, __nv_bfloat16* dst) {
    const uint4 a = *reinterpret_cast<const uint4*>(src + c * 8);
    const uint4 b = *reinterpret_cast<const uint4*>(src + HALF + c * 8);
    float x1[8], x2[8];
    unpack8(a, x1);
    unpack8(b, x2);
    uint32_t y1[4], y2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e0 = 2 * i, e1 = 2 * i + 1;
      y1[i] = pack_bf16(x1[e0] * cs[e0] - x2[e0] * sn[e0], x1[e1] * cs[e1] - x2[e1] * sn[e1]);
      y2[i] = pack_bf16(x2[e0] * cs[e0] + x1[e0] * sn[e0], x2[e1] * cs[e1] + x1[e1] * sn[e1]);
    }
    *reinterpret_cast<uint4*>(dst + c * 8) = make_uint4(y1[0], y1[1], y1[2], y1[3]);
    *reinterpret_cast<uint4*>(dst + HALF + c * 8) = make_uint4(y2[0], y2[1], y2[2], y2[3]);
  };
  // this thread's heads [h0, h1) of the combined list: its Q heads, then its K heads
  const int h0 = grp * p.hpt, h1 = min(h0 + p.hpt, H);
  const int qe = min(h1, p.Hq);
#pragma unroll 4
  for (int h = h0; h < qe; ++h)
    rotate(p.q + t * p.qs + (int64_t)h * D, p.qo + t * p.qos + (int64_t)h * D);
#pragma unroll 4
  for (int h = max(h0, p.Hq); h < h1; ++h)
    rotate(p.k + t * p.ks + (int64_t)(h - p.Hq) * D, p.ko + t * p.kos + (int64_t)(h - p.Hq) * D);
}

// K at the reused position ids of a plan: one block per query tile of the
// plan's work list (the tiles partition every request's rows), so a row's
// request and set start come from the plan: rows of the shared set sit at
// j - s0, row j of an item set starting at a at S + (j - a).
struct RopePlanParams {
  const ReqInfo* req;
  const int32_t* seg_start;
  const WorkItem* units;
  int32_t qbase;
  const __nv_bfloat16* k;
  __nv_bfloat16* ko;
  int64_t ks, kos;
  int32_t Hkv;
  float inv_freq[64];
};

template <int D>
__global__ void __launch_bounds__(kRopeThreads)
mis_rope_k_plan_kernel(const RopePlanParams p) {
  griddep_wait();                                     // no early trigger (see mis_rope_kernel)
  constexpr int HALF = D / 2, NC = HALF / 8;          // 8-pair chunks per head
  const WorkItem un = p.units[blockIdx.x];
  const ReqInfo R = p.req[un.req];
  // gridDim.y blocks share a tile (few tiles: more blocks than tiles)
  const int stride = blockDim.x * gridDim.y;
  for (int cell = threadIdx.x + blockDim.x * blockIdx.y; cell < kBM * NC; cell += stride) {
    const int c = cell % NC, j = un.q0 + cell / NC;
    if (j >= R.e0) break;                             // cells run row by row
    const int jn = j - p.qbase;
    const int pos = j < R.pend ? j - R.s0 : (R.pend - R.s0) + (j - p.seg_start[jn]);
    const float fp = (float)pos;
    float cs[8], sn[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) sincosf(fp * p.inv_freq[c * 8 + e], &sn[e], &cs[e]);
    for (int h = 0; h < p.Hkv; ++h) {
      const __nv_bfloat16* src = p.k + jn * p.ks + (int64_t)h * D;
      __nv_bfloat16* dst = p.ko + jn * p.kos + (int64_t)h * D;
      const uint4 a = *reinterpret_cast<const uint4*>(src + c * 8);
      const uint4 b = *reinterpret_cast<const uint4*>(src + HALF + c * 8);
      float x1[8], x2[8];
      unpack8(a, x1);
      unpack8(b, x2);
      uint32_t y1[4], y2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e0 = 2 * i, e1 = 2 * i + 1;
        y1[i] = pack_bf16(x1[e0] * cs[e0] - x2[e0] * sn[e0], x1[e1] * cs[e1] - x2[e1] * sn[e1]);
        y2[i] = pack_bf16(x2[e0] * cs[e0] + x1[e0] * sn[e0], x2[e1] * cs[e1] + x1[e1] * sn[e1]);
      }
      *reinterpret_cast<uint4*>(dst + c * 8) = make_uint4(y1[0], y1[1], y1[2], y1[3]);
      *reinterpret_cast<uint4*>(dst + HALF + c * 8) = make_uint4(y2[0], y2[1], y2[2], y2[3]);
    }
  }
}

template <int D>
mis_status_t launch_rope_d(RopeParams& p, double base, cudaStream_t st) {
  for (int i = 0; i < D / 2; ++i) p.inv_freq[i] = (float)std::pow(base, -2.0 * i / D);
  const int64_t H = p.Hq + p.Hkv, cells = (int64_t)p.T * (D / 16);   // (row, chunk) pairs
  // split the heads of a row over several threads only while the (row, chunk)
  // cells alone would fill less than half of the target
  const int64_t want = kThreadsPerSm * num_sms();
  const int64_t split = std::max<int64_t>(1, std::min<int64_t>(H, want / (2 * cells)));
  p.hpt = (int32_t)((H + split - 1) / split);
  const int64_t groups = (H + p.hpt - 1) / p.hpt;
  const int64_t threads = cells * groups;
  const int64_t blocks = (threads + kRopeThreads - 1) / kRopeThreads;
  if (blocks > 0x7fffffff) return MIS_ERR_UNSUPPORTED;
  return launch_pdl(mis_rope_kernel<D>, dim3((unsigned)blocks), dim3(kRopeThreads), 0, st, p) ==
                 cudaSuccess
             ? MIS_OK
             : MIS_ERR_CUDA;
}

}  // namespace
}  // namespace mis

extern "C" mis_status_t mis_rope_qk(const void* q, const void* k, void* q_out, void* k_out,
                                    int64_t q_row_stride, int64_t k_row_stride,
                                    int64_t q_out_row_stride, int64_t k_out_row_stride, int32_t T,
                                    int32_t Hq, int32_t Hkv, int32_t D,
                                    const int32_t* position_ids, double base, void* stream) {
  using namespace mis;
  if (T < 0 || Hq < 1 || Hkv < 1) return MIS_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return MIS_ERR_UNSUPPORTED;
  if (!(base > 1.0) || !std::isfinite(base)) return MIS_ERR_INVALID_ARG;
  if (T == 0) return MIS_OK;
  // q and q_out both null: K only (Q is rotated on load by the attention call)
  if ((q == nullptr) != (q_out == nullptr)) return MIS_ERR_INVALID_ARG;
  const bool with_q = q != nullptr;
  if (!k || !k_out || !position_ids) return MIS_ERR_INVALID_ARG;
  auto misaligned = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  if (misaligned(q) || misaligned(k) || misaligned(q_out) || misaligned(k_out))
    return MIS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(position_ids) & 3u) return MIS_ERR_INVALID_ARG;
  const int64_t wq = (int64_t)Hq * D, wk = (int64_t)Hkv * D;
  if (with_q && (q_row_stride < wq || q_out_row_stride < wq || ((q_row_stride | q_out_row_stride) & 7)))
    return MIS_ERR_SHAPE;
  if (k_row_stride < wk || k_out_row_stride < wk || ((k_row_stride | k_out_row_stride) & 7))
    return MIS_ERR_SHAPE;
  if (!with_q) Hq = 0;                  // the kernel's head list holds the K heads only
  RopeParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.qo = static_cast<__nv_bfloat16*>(q_out);
  p.ko = static_cast<__nv_bfloat16*>(k_out);
  p.qs = q_row_stride; p.ks = k_row_stride; p.qos = q_out_row_stride; p.kos = k_out_row_stride;
  p.pos = position_ids;
  p.T = T; p.Hq = Hq; p.Hkv = Hkv;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  try {
    return D == 128 ? launch_rope_d<128>(p, base, st) : launch_rope_d<64>(p, base, st);
  } catch (...) {
    return MIS_ERR_CUDA;
  }
}


extern "C" mis_status_t mis_rope_k_plan(mis_plan_t plan, const void* k, void* k_out,
                                        int64_t k_row_stride, int64_t k_out_row_stride,
                                        double base, void* stream) {
  using namespace mis;
  if (!plan) return MIS_ERR_INVALID_ARG;
  const HostPlan& pl = plan_of(plan);
  if (!pl.workspace) return MIS_ERR_WORKSPACE;
  if (!k || !k_out) return MIS_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(k_out)) & 15u)
    return MIS_ERR_INVALID_ARG;
  if (!(base > 1.0) || !std::isfinite(base)) return MIS_ERR_INVALID_ARG;
  const int64_t wk = (int64_t)pl.Hkv * pl.D;
  if (k_row_stride < wk || k_out_row_stride < wk || ((k_row_stride | k_out_row_stride) & 7))
    return MIS_ERR_SHAPE;
  if (pl.work.empty()) return MIS_OK;
  if (pl.work.size() > 0x7fffffff) return MIS_ERR_UNSUPPORTED;
  const uint8_t* ws = static_cast<const uint8_t*>(pl.workspace);
  RopePlanParams p;
  p.req = reinterpret_cast<const ReqInfo*>(ws + pl.off_req);
  p.seg_start = reinterpret_cast<const int32_t*>(ws + pl.off_seg);
  p.units = reinterpret_cast<const WorkItem*>(ws + pl.off_work);
  p.qbase = pl.cached ? pl.qbase : 0;
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.ko = static_cast<__nv_bfloat16*>(k_out);
  p.ks = k_row_stride; p.kos = k_out_row_stride;
  p.Hkv = pl.Hkv;
  for (int i = 0; i < 64; ++i)
    p.inv_freq[i] = i < pl.D / 2 ? (float)std::pow(base, -2.0 * i / pl.D) : 0.f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // at least about four blocks per SM: a tile's 128 rows split over up to 4 blocks
  const int64_t tiles = (int64_t)pl.work.size();
  const int64_t ysplit = std::min<int64_t>(4, std::max<int64_t>(1, (4 * num_sms() + tiles - 1) / tiles));
  const dim3 grid((unsigned)tiles, (unsigned)ysplit);
  try {
    const cudaError_t e = pl.D == 128
        ? launch_pdl(mis_rope_k_plan_kernel<128>, grid, dim3(kRopeThreads), 0, st, p)
        : launch_pdl(mis_rope_k_plan_kernel<64>, grid, dim3(kRopeThreads), 0, st, p);
    return e == cudaSuccess ? MIS_OK : MIS_ERR_CUDA;
  } catch (...) {
    return MIS_ERR_CUDA;
  }
}
