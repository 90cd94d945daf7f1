// MIS attention forward for sm_103a.
//
// Computes O_j = softmax(scale * q_j K_A^T) V_A over the keys A(j) visible
// from row j under eq. (4) of "From Generation to Scoring: Scaling LLM-Based
// Semantic Labeling at LinkedIn" (Section 4.1): the shared rows Q attend
// causally, rows of item i attend to all of Q and causally inside I_i. The
// host planner lists, per 128-row query tile, only the 128-key tiles that hold
// a visible entry and flags the ones that need the element mask, so masked
// item x item blocks are never loaded or multiplied ("Turbocharging LinkedIn's
// recommendation systems with SGLang", "Implemented skip tiles"; Section 4.2
// of the former: attention work O(Lq^2 + N Lq Lbar) instead of the causal
// O((Lq + N Lbar)^2)).
//
// One block = one (query tile, query head). Warp roles:
//   warp 0     : TMA producer (Q once, then K/V tiles through a ring of stages)
//   warp 1     : TMEM allocator and the single thread that issues tcgen05.mma
//                  S = Q K^T  (SS: both operands in shared memory)
//                  O += P V   (TS: P from tensor memory, V in shared memory)
//   warps 4..7 : softmax, one TMEM lane (= one query row) per thread; the row
//                max and sum stay inside the thread, so no shuffles are needed.
// Tensor memory (512 columns): S0 | S1 | O | P0 | P1. S is double buffered so
// the tensor core computes S_{t+1} while the softmax works on S_t.
// The running maximum is only moved (and O rescaled in TMEM) when it grows by
// more than 2^8; the final division by the row sum makes the result exact for
// any reference maximum.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>

#include "mis_internal.h"
#include "mis_ptx.cuh"

namespace mis {

CUtensorMap make_tmap_bf16(const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box, bool* ok);

namespace {

using namespace dev;

template <int D>
struct AttnCfg {
  static constexpr int kStages = (D == 128) ? 3 : 4;
  static constexpr int kBox = kBN * 64 * 2;            // one 64-column box, 128 rows: 16 KB
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kTile = kBN * D * 2;            // K or V tile
  static constexpr int kStageBytes = 2 * kTile;
  static constexpr int kData = kQBytes + kStages * kStageBytes;
  static constexpr int kSmem = kData + 512 + 1024;     // barriers + alignment slack
};

constexpr uint32_t kColS0 = 0, kColO = 256, kColP0 = 384;
constexpr float kRescaleThreshold = 8.0f;             // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

struct AttnParams {
  const ReqInfo* req;
  const int32_t* seg_start;
  const WorkItem* work;
  const uint32_t* klist;
  __nv_bfloat16* o;
  float* lse;
  int64_t o_stride;
  int32_t T;
  int32_t group;        // Hq / Hkv
  float scale_log2;     // softmax scale * log2(e)
  uint32_t* status;
  uint64_t wait_ns;
};

template <int D>
__global__ void __launch_bounds__(256, 1)
mis_attn_fwd_kernel(const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const AttnParams p) {
  using C = AttnCfg<D>;
  constexpr int NS = C::kStages;
  constexpr int NB = D / 64;                          // 64-column boxes per row
  // barrier slots
  constexpr int bQ = 0, bKVF = 1, bKVE = bKVF + NS, bSF = bKVE + NS, bPF = bSF + 2,
                bOD = bPF + 2, bDR = bOD + 1, nBar = bDR + 1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::kQBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kData);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + nBar);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* skip_flag = tmem_slot + 2;
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WorkItem wi = p.work[blockIdx.x];
  const int h = blockIdx.y;
  const int g = h / p.group;
  const ReqInfo R = p.req[wi.req];
  const int nk = wi.nk;

  if (threadIdx.x == 0) {
    *skip_flag = (*(volatile uint32_t*)p.status & kDevTimeout) ? 1u : 0u;
    *abort_flag = 0;
    mbar_init(bar(bQ), 1);
    for (int s = 0; s < NS; ++s) { mbar_init(bar(bKVF + s), 1); mbar_init(bar(bKVE + s), 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(bar(bSF + s), 1); mbar_init(bar(bPF + s), 128); }
    mbar_init(bar(bOD), 1);
    mbar_init(bar(bDR), 1);
    fence_mbar_init();
    fence_proxy_async();
  }
  __syncthreads();
  if (*skip_flag) return;                 // another block already gave up
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{abort_flag, p.status, p.wait_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&qmap); tma_prefetch_desc(&kmap); tma_prefetch_desc(&vmap);
      mbar_arrive_expect_tx(bar(bQ), C::kQBytes);
      for (int b = 0; b < NB; ++b)
        tma_load_3d(smem_u32(sQ + b * C::kBox), &qmap, bar(bQ), b * 64, h, wi.q0);
      int issued = 0;
      for (int it = 0; it < nk; ++it) {
        const int st = it % NS;
        if (it >= NS && !wait(bar(bKVE + st), ((it / NS) - 1) & 1, W, 0x100 + it)) break;
        const int32_t c0 = (int32_t)(p.klist[wi.kofs + it] & ~kNeedMask);
        uint8_t* sK = sKV + st * C::kStageBytes;
        uint8_t* sV = sK + C::kTile;
        mbar_arrive_expect_tx(bar(bKVF + st), C::kStageBytes);
        for (int b = 0; b < NB; ++b) {
          tma_load_3d(smem_u32(sK + b * C::kBox), &kmap, bar(bKVF + st), b * 64, g, c0);
          tma_load_3d(smem_u32(sV + b * C::kBox), &vmap, bar(bKVF + st), b * 64, g, c0);
        }
        issued = it + 1;
      }
      // drain: every copy this thread started has landed before the block exits
      wait_drain(bar(bQ), 0);
      for (int i = (issued > NS ? issued - NS : 0); i < issued; ++i)
        wait_drain(bar(bKVF + i % NS), (i / NS) & 1);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16(128, kBN, false);
      constexpr uint32_t idO = idesc_bf16(128, D, true);
      const uint32_t aQ = smem_u32(sQ);
      bool ok = wait(bar(bQ), 0, W, 0x200);
      auto issue_s = [&](int it) -> bool {
        const int st = it % NS;
        if (!wait(bar(bKVF + st), (it / NS) & 1, W, 0x300 + it)) return false;
        tc_fence_after();
        const uint32_t aK = smem_u32(sKV + st * C::kStageBytes);
        const uint32_t dS = tmem + kColS0 + (it & 1) * 128;
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t da = sdesc_sw128(aQ + b * C::kBox + ks * 32, 16, 1024);
            const uint64_t db = sdesc_sw128(aK + b * C::kBox + ks * 32, 16, 1024);
            mma_ss(dS, da, db, idS, (b | ks) != 0);
          }
        mma_commit(bar(bSF + (it & 1)));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int it = 0; ok && it < nk; ++it) {
        if (it + 1 < nk && !issue_s(it + 1)) break;
        if (!wait(bar(bPF + (it & 1)), (it >> 1) & 1, W, 0x400 + it)) break;
        tc_fence_after();
        const int st = it % NS;
        const uint32_t aV = smem_u32(sKV + st * C::kStageBytes + C::kTile);
        const uint32_t aP = tmem + kColP0 + (it & 1) * 64;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          // V is MN-major (head dim contiguous): 8-key groups 1024 B apart,
          // 64-column boxes kBox apart.
          const uint64_t db = sdesc_sw128(aV + ks * 16 * 128, C::kBox, 1024);
          mma_ts(tmem + kColO, aP + ks * 8, db, idO, (it | ks) != 0);
        }
        mma_commit(bar(bKVE + st));
        mma_commit(bar(bOD));
      }
      // drain: all tensor-core work of this thread completes before dealloc
      mma_commit(bar(bDR));
      wait_drain(bar(bDR), 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------- softmax
    const int sw = warp - 4;
    const int r = sw * 32 + lane;
    const int j = wi.q0 + r;
    const bool valid = j < R.e0;
    const int jj = valid ? j : -1;                    // invalid rows see nothing
    const int lo = valid ? p.seg_start[j] : 0x7fffffff;
    const uint32_t tl = tmem + ((uint32_t)(sw * 32) << 16);
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int it = 0; it < nk; ++it) {
      const uint32_t e = p.klist[wi.kofs + it];
      const int32_t c0 = (int32_t)(e & ~kNeedMask);
      const int b = it & 1;
      ok = wait(bar(bSF + b), (it >> 1) & 1, W, 0x500 + it);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t su[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) tmem_ld32(tl + kColS0 + b * 128 + c * 32, su + c * 32);
      tmem_ld_wait();
      if (e & kNeedMask) {
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          const int k = c0 + c;
          const bool vis = (k <= jj) && (k < R.pend || k >= lo);
          su[c] = vis ? su[c] : 0xff800000u;          // -inf
        }
      }
      float mx = __uint_as_float(su[0]);
#pragma unroll
      for (int c = 1; c < kBN; ++c) mx = fmaxf(mx, __uint_as_float(su[c]));
      const float m_new = fmaxf(m_ref, mx * sl2);
      const bool grow = m_new > m_ref + kRescaleThreshold;
      // PV of the previous tile must be done before O is touched; waiting on
      // every completion in turn also keeps this barrier's parity in step.
      if (it > 0) {
        ok = wait(bar(bOD), (it - 1) & 1, W, 0x600 + it);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      if (__any_sync(0xffffffffu, grow)) {
        const float alpha = grow ? ex2(m_ref - m_new) : 1.f;
        if (it > 0) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tl + kColO + c * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * alpha);
            tmem_st32(tl + kColO + c * 32, ov);
          }
          tmem_st_wait();
        }
        if (grow) { l *= alpha; m_ref = m_new; }
      }
      const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;
      float rs = 0.f;
      uint32_t pk[kBN / 2];
#pragma unroll
      for (int c = 0; c < kBN / 2; ++c) {
        const float p0 = ex2(fmaf(__uint_as_float(su[2 * c]), sl2, -mb));
        const float p1 = ex2(fmaf(__uint_as_float(su[2 * c + 1]), sl2, -mb));
        rs += p0 + p1;
        pk[c] = pack_bf16(p0, p1);
      }
      l += rs;
#pragma unroll
      for (int c = 0; c < kBN / 64; ++c)
        tmem_st32(tl + kColP0 + b * 64 + c * 32, pk + c * 32);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar(bPF + b));
    }
    if (ok) {
      ok = wait(bar(bOD), (nk - 1) & 1, W, 0x700);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.o + (int64_t)(valid ? j : 0) * p.o_stride + (int64_t)h * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tmem_ld32(tl + kColO + c * 32, ov);
        tmem_ld_wait();
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(ov[8 * q + 0]) * inv, __uint_as_float(ov[8 * q + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(ov[8 * q + 2]) * inv, __uint_as_float(ov[8 * q + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(ov[8 * q + 4]) * inv, __uint_as_float(ov[8 * q + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(ov[8 * q + 6]) * inv, __uint_as_float(ov[8 * q + 7]) * inv);
            dst[q] = w;
          }
        }
      }
      if (p.lse && valid) p.lse[(int64_t)h * p.T + j] = (m_ref + log2f(l)) * kLn2;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
mis_status_t launch_d(const HostPlan& pl, const void* q, const void* k, const void* v, void* o,
                      float* lse, int64_t qs, int64_t ks, int64_t vs, int64_t os, void* stream) {
  using C = AttnCfg<D>;
  bool ok = true;
  const uint32_t box[3] = {64, 1, (uint32_t)kBM};
  const uint64_t qd[3] = {(uint64_t)D, (uint64_t)pl.Hq, (uint64_t)pl.T};
  const uint64_t qstr[2] = {(uint64_t)D * 2, (uint64_t)qs * 2};
  const uint64_t kd[3] = {(uint64_t)D, (uint64_t)pl.Hkv, (uint64_t)pl.T};
  const uint64_t kstr[2] = {(uint64_t)D * 2, (uint64_t)ks * 2};
  const uint64_t vstr[2] = {(uint64_t)D * 2, (uint64_t)vs * 2};
  CUtensorMap qm = make_tmap_bf16(q, 3, qd, qstr, box, &ok);
  CUtensorMap km = make_tmap_bf16(k, 3, kd, kstr, box, &ok);
  CUtensorMap vm = make_tmap_bf16(v, 3, kd, vstr, box, &ok);
  if (!ok) return MIS_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(pl.workspace);
  AttnParams prm;
  prm.req = reinterpret_cast<const ReqInfo*>(ws + pl.off_req);
  prm.seg_start = reinterpret_cast<const int32_t*>(ws + pl.off_seg);
  prm.work = reinterpret_cast<const WorkItem*>(ws + pl.off_work);
  prm.klist = reinterpret_cast<const uint32_t*>(ws + pl.off_klist);
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.o_stride = os;
  prm.T = pl.T;
  prm.group = pl.Hq / pl.Hkv;
  prm.scale_log2 = pl.scale * 1.4426950408889634f;
  prm.status = reinterpret_cast<uint32_t*>(ws);
  prm.wait_ns = wait_limit_ns();

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, 8, st) != cudaSuccess) return MIS_ERR_CUDA;
  if (pl.work.empty()) return MIS_OK;
  auto kern = mis_attn_fwd_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) !=
      cudaSuccess)
    return MIS_ERR_CUDA;
  dim3 grid((unsigned)pl.work.size(), (unsigned)pl.Hq);
  kern<<<grid, 256, C::kSmem, st>>>(qm, km, vm, prm);
  return cudaGetLastError() == cudaSuccess ? MIS_OK : MIS_ERR_CUDA;
}

}  // namespace

mis_status_t launch_attention(const HostPlan& p, const void* q, const void* k, const void* v,
                              void* o, float* lse, int64_t qs, int64_t ks, int64_t vs, int64_t os,
                              void* stream) {
  if (p.D == 128) return launch_d<128>(p, q, k, v, o, lse, qs, ks, vs, os, stream);
  if (p.D == 64) return launch_d<64>(p, q, k, v, o, lse, qs, ks, vs, os, stream);
  return MIS_ERR_UNSUPPORTED;
}

}  // namespace mis
