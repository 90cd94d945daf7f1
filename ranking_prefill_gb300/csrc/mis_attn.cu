// MIS attention forward for sm_103a.
//
// Computes O_j = softmax(scale * q_j K_A^T) V_A over the keys A(j) visible
// from row j under eq. (4) of "From Generation to Scoring: Scaling LLM-Based
// Semantic Labeling at LinkedIn" (Section 4.1): the shared rows Q attend
// causally, rows of item i attend to all of Q and causally inside I_i. The
// host planner lists, per 128-row query tile, only the 128-key tiles that hold
// a visible entry and flags the ones that need the element mask, so masked
// item x item blocks are never loaded or multiplied ("Turbocharging LinkedIn's
// recommendation systems with SGLang", section "FlashInfer changes"; Section
// 4.2 of "From Generation to Scoring": attention work O(Lq^2 + N Lq Lbar)
// instead of the causal O((Lq + N Lbar)^2)).
//
// Persistent kernel: one block per SM walks the planner's units in
// longest-first order, snaking over the blocks. A unit is a query tile with
// its key-tile list and either
//   * a pair of query heads that share a kv head ("pair" schedule): stream t
//     of the block computes head t over every key tile, or
//   * one query head ("split" schedule): stream t takes the key tiles
//     t, t+2, t+4, ... of that head, and the two partial results (running
//     maximum, row sum, unnormalised O) are merged in the epilogue.
// The split schedule doubles the number of units and halves their length,
// which the planner picks when the pair units would leave the last wave of
// blocks half empty, and always for odd GQA group sizes. Pipelines, barriers
// and tensor memory carry over from unit to unit: the next unit's Q and first
// K/V tiles load while the current one finishes, and its first S product
// runs during the epilogue.
//
// Warp roles (512 threads, four warpgroups):
//   warp 0      : TMA producer (the unit's Q tiles, then K and V tiles
//                 through separate rings: K is released once its S products
//                 are issued, V after its PV products)
//   warp 1      : TMEM allocator and the single thread issuing tcgen05.mma:
//                   S_t = Q K^T  (SS: both operands in shared memory)
//                   O_t += P_t V (TS: P_t from tensor memory, V MN-major)
//                 in the order S_0(s), PV_1(s-1), S_1(s), PV_0(s) for step s,
//                 so each stream's softmax overlaps the other's products
//   warps 4..7  : softmax of stream 0, warps 8..11: of stream 1. One TMEM
//                 lane (= one query row) per thread: the row max and sum stay
//                 in the thread, no shuffles. At the end of a unit a thread
//                 leaves its row's (max, sum) in shared memory and moves on to
//                 the next unit's first S tile at once.
//   warps 12..15: epilogue. Once every PV of the unit is done they read O out
//                 of tensor memory (handing each accumulator back to the MMA
//                 thread as soon as it is read), merge the split schedule's
//                 two partial results, normalise, and store O (and the LSE).
//                 The epilogue of unit u thus overlaps the first softmax of
//                 unit u+1 instead of delaying it.
// Registers are rebalanced per warpgroup after the prologue (setmaxnreg):
// the softmax warpgroups hold a whole 128-column S row per thread.
// Tensor memory (512 columns): S_0 | S_1 | O_0 | O_1. P_t (bf16 pairs) is
// written over the first half of S_t once S_t has been read. Because S_t(s)
// is committed after PV_t(s-1) was issued, "S_t(s) ready" also means O_t and
// the previous P_t are free, so the softmax never waits on a PV.
// The running maximum is only moved (and O rescaled in TMEM) when it grows by
// more than 2^8; the final division by the row sum makes the result exact for
// any reference maximum, and the same holds for the merge of the split
// schedule's two partial results.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "mis_internal.h"
#include "mis_ptx.cuh"

namespace mis {

CUtensorMap make_tmap_bf16(const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box, bool* ok);

namespace {

using namespace dev;

template <int D>
struct AttnCfg {
  static constexpr int kBox = kBN * 64 * 2;            // one 64-column box, 128 rows: 16 KB
  static constexpr int kTile = kBN * D * 2;            // a Q, K or V tile
  static constexpr int kKStages = (D == 128) ? 2 : 4;
  static constexpr int kVStages = (D == 128) ? 2 : 4;
  static constexpr int kOWarp = 32 * 128;              // O staging per epilogue warp: 32 rows x 64 bf16
  static constexpr int kStats = 2 * 2 * kBM * 8;       // (max, sum) per row: 2 slots x 2 streams
  static constexpr int kData = (2 + kKStages + kVStages) * kTile + 4 * kOWarp + kStats;
  static constexpr int kSmem = kData + 512 + 1024;     // barriers + alignment slack
};

constexpr int kThreads = 512;
// Per-thread register budgets after the prologue (control, epilogue, softmax
// warpgroups); 128 + 128 + 256 threads must fit the launch's 512 x 128. The
// split schedule's softmax keeps a few more values live, its epilogue merges
// in 16-column pieces.
template <bool kSplit>
struct RegSplit {
  static constexpr int kCtl = kSplit ? 80 : 88;
  static constexpr int kEpi = kSplit ? 64 : 72;
  static constexpr int kSoftmax = kSplit ? 184 : 176;
  static_assert(128 * kCtl + 128 * kEpi + 256 * kSoftmax <= kThreads * 128,
                "register split exceeds the launch allocation");
};
constexpr float kRescaleThreshold = 8.0f;             // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

struct AttnParams {
  const ReqInfo* req;
  const int32_t* seg_start;
  const WorkItem* units;  // query tiles, longest first
  const uint32_t* klist;
  int32_t n_units;        // query tiles
  const int32_t* order;   // or null: the unit at each walk position (-1: none), see unit_at
  int32_t n_walk;         // walk positions (units in all when there is no order)
  __nv_bfloat16* o;
  float* lse;
  int64_t o_stride;
  int32_t T;
  int32_t qbase;          // virtual row of new row 0 (0 unless the plan reads a prefix cache)
  int32_t group;          // Hq / Hkv
  int32_t n_head_groups;  // units per query tile: Hq / 2 (pair) or Hq (split)
  float scale_log2;       // softmax scale * log2(e)
  uint32_t* status;
  uint64_t wait_ns;
  uint32_t stall;         // failure injection: wait on a barrier nothing arrives on
  // rotary embedding of Q on load (rope == 0: Q arrives rotated)
  int32_t rope;
  float rope_freq[64];      // base^(-2i/D), i < D/2 (fp64 on the host, rounded to fp32)
};

// sin and cos of x (|x| < 2^16 * pi): x is reduced to r in [-pi, pi] by the
// Cody-Waite method (2 pi split into a high part exact in 8 bits, so k * high
// is exact for k < 2^16, and the fp32 remainder), then the SFU's sin/cos
// approximations, whose absolute error on [-pi, pi] is about 2^-21.
__device__ __forceinline__ void sincos_reduced(float x, float& sn, float& cs) {
  constexpr float kInv2Pi = 0.15915494309189535f;
  constexpr float k2PiHi = 6.28125f;                          // 201 / 32
  constexpr float k2PiLo = 0.0019353071795864769f;            // 2 pi - 6.28125
  const float k = rintf(x * kInv2Pi);
  const float r = fmaf(-k, k2PiLo, fmaf(-k, k2PiHi, x));
  asm("sin.approx.f32 %0, %1;" : "=f"(sn) : "f"(r));
  asm("cos.approx.f32 %0, %1;" : "=f"(cs) : "f"(r));
}

// Rotary embedding of ROWS rows of NH Q tiles (heads at the same rows) in
// shared memory, in place, by one warp. A tile is NB boxes of 128 rows x 64
// bf16 columns with the 128-byte swizzle (16-byte chunk c of row r at chunk
// c ^ (r & 7)); tile h starts kTileBytes after tile h - 1. Rotate-half form:
// the pair (x[i], x[i + D/2]) turns by the angle of frequency i. A "chunk
// pair" g holds frequencies 8g .. 8g+7 (one 16-byte chunk of each half);
// this warp turns the chunk pairs g0, g0 + GS, ... of rows r0 .. r0+ROWS-1.
// Lanes are laid out (row, chunk pair), so a warp's shared-memory accesses
// cover whole tile rows, and each angle is computed once for the NH heads.
template <int D, int GS, int NH, int ROWS>
struct RopeWarp {
  static constexpr int kCpr = D / 16 / GS;   // chunk pairs of a row this warp turns
  static constexpr int kRpp = 32 / kCpr;     // rows per pass
  static constexpr int kPasses = ROWS / kRpp;
  static constexpr int kTileBytes = kBM * D * 2;
  static_assert(ROWS % kRpp == 0, "rows per warp");
  float4 cs[kPasses][4];   // (cos, sin, cos, sin) of the lane's 8 frequencies, per pass

  // The angles of every pass, computed while the tiles land. pos: the
  // position of row r0 + lane % ROWS, or -1 (row outside the request: the
  // identity).
  __device__ __forceinline__ void angles(const float* freq, int pos, int g0) {
    const int lane = threadIdx.x & 31;
    const int g = g0 + lane % kCpr * GS;
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = freq[8 * g + e];
#pragma unroll
    for (int k = 0; k < kPasses; ++k) {
      const int pk = __shfl_sync(0xffffffffu, pos, k * kRpp + lane / kCpr);
      const float fp = (float)max(pk, 0);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        float s0, c0, s1, c1;
        sincos_reduced(fp * f[2 * w], s0, c0);
        sincos_reduced(fp * f[2 * w + 1], s1, c1);
        cs[k][w] = pk >= 0 ? make_float4(c0, s0, c1, s1) : make_float4(1.f, 0.f, 1.f, 0.f);
      }
    }
  }

  __device__ __forceinline__ void turn(uint32_t sq, int r0, int g0) const {
    constexpr int HALF = D / 2, BOX = kBN * 64 * 2;
    const int lane = threadIdx.x & 31;
    const int g = g0 + lane % kCpr * GS;
    const int c1 = 8 * g, c2 = 8 * g + HALF;
#pragma unroll
    for (int k = 0; k < kPasses; ++k) {
      const int r = r0 + k * kRpp + lane / kCpr;
      const uint32_t row = sq + (uint32_t)r * 128u;
      const int sw = r & 7;
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        const uint32_t a1 = row + (uint32_t)(h * kTileBytes + (c1 >> 6) * BOX) +
                            ((((c1 & 63) >> 3) ^ sw) << 4);
        const uint32_t a2 = row + (uint32_t)(h * kTileBytes + (c2 >> 6) * BOX) +
                            ((((c2 & 63) >> 3) ^ sw) << 4);
        uint32_t x[4], y[4];
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]) : "r"(a1) : "memory");
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(y[0]), "=r"(y[1]), "=r"(y[2]), "=r"(y[3]) : "r"(a2) : "memory");
        uint32_t ox[4], oy[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float4 c = cs[k][w];                 // frequencies 8g + 2w, 8g + 2w + 1
          const float x0 = __uint_as_float(x[w] << 16), x1 = __uint_as_float(x[w] & 0xffff0000u);
          const float y0 = __uint_as_float(y[w] << 16), y1 = __uint_as_float(y[w] & 0xffff0000u);
          ox[w] = pack_bf16(fmaf(x0, c.x, -y0 * c.y), fmaf(x1, c.z, -y1 * c.w));
          oy[w] = pack_bf16(fmaf(y0, c.x, x0 * c.y), fmaf(y1, c.z, x1 * c.w));
        }
        st_shared_v4(a1, ox[0], ox[1], ox[2], ox[3]);
        st_shared_v4(a2, oy[0], oy[1], oy[2], oy[3]);
      }
    }
  }
};

// Unit handled by this block in pass kk: walk position kk * G + c, passes
// alternating direction (snake order), so over the longest-first unit list
// every block gets a long and a short unit from each pair of passes. A plan
// may instead give the unit at every walk position (a greedy assignment in
// list order that balances the blocks better, e.g. over many requests whose
// units are ordered request by request); -1 = none at that position.
__device__ __forceinline__ int unit_at(const AttnParams& p, int kk) {
  const int G = gridDim.x, c = blockIdx.x;
  const int pos = kk * G + ((kk & 1) ? (G - 1 - c) : c);
  if (pos >= p.n_walk) return -1;
  return p.order ? p.order[pos] : pos;
}

template <int D, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
mis_attn_fwd_kernel(const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap,
                    const __grid_constant__ CUtensorMap omap,
                    const __grid_constant__ CUtensorMap kcmap,
                    const __grid_constant__ CUtensorMap vcmap, const AttnParams p) {
  using C = AttnCfg<D>;
  constexpr int KS = C::kKStages, VS = C::kVStages;
  constexpr int NB = D / 64;                          // 64-column boxes per row
  // TMEM columns: S_t at 128 t, O_t at 256 + D t
  auto colS = [](int t) { return (uint32_t)(t * 128); };
  auto colO = [](int t) { return (uint32_t)(256 + t * D); };
  // barrier slots
  //   ST_{s,t}: stream t's (max, sum) of a unit written to stats slot s;
  //   SE_s: the epilogue has read slot s
  constexpr int bQF = 0, bQE = 1, bKF = 2, bKE = bKF + KS, bVF = bKE + KS, bVE = bVF + VS,
                bSF = bVE + VS, bPF = bSF + 2, bOF = bPF + 2, bOE = bOF + 1, bDR = bOE + 2,
                bST = bDR + 1, bSE = bST + 4, bQR = bSE + 2, nBar = bQR + 1;
  // bQR: the unit's Q tiles rotated in place (rotary embedding on load)

  griddep_launch_dependents();

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem;                                  // 2 tiles
  uint8_t* sK = smem + 2 * C::kTile;                   // KS tiles
  uint8_t* sV = sK + KS * C::kTile;                    // VS tiles
  uint8_t* sO = sV + VS * C::kTile;                    // 4 x kOWarp: O staging of the epilogue warps
  // (max, sum) of every row at the end of a unit: [slot = unit & 1][stream][row]
  float2* stats = reinterpret_cast<float2*>(sO + 4 * C::kOWarp);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kData);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + nBar);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* skip_flag = tmem_slot + 2;
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool split = kSplit;
  constexpr int nh = split ? 1 : 2;                    // Q tiles (heads) per unit
  const int n_hg = p.n_head_groups;
  const int total = p.n_walk;                          // walk positions; unit u: p.units[u / n_hg], head group u % n_hg

  // prologue (shared memory and tensor memory only) overlaps the previous
  // kernel in the stream; global memory is read after griddepcontrol.wait
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(bQF), 1);
    mbar_init(bar(bQE), 1);
    for (int s = 0; s < KS; ++s) { mbar_init(bar(bKF + s), 1); mbar_init(bar(bKE + s), 1); }
    for (int s = 0; s < VS; ++s) { mbar_init(bar(bVF + s), 1); mbar_init(bar(bVE + s), 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(bSF + s), 1);
      mbar_init(bar(bPF + s), 4);                      // one arrival per softmax warp
      mbar_init(bar(bOE + s), 4);                      // one arrival per epilogue warp
      mbar_init(bar(bST + 2 * s), kBM);                // every thread of stream 0
      mbar_init(bar(bST + 2 * s + 1), kBM);            // ... of stream 1
      mbar_init(bar(bSE + s), kBM);                    // every epilogue thread
    }
    mbar_init(bar(bOF), 1);
    mbar_init(bar(bDR), 1);
    mbar_init(bar(bQR), 8);                            // one arrival per softmax warp
    fence_mbar_init();
    fence_proxy_async();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&qmap); tma_prefetch_desc(&kmap); tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&omap);
    if (p.qbase) { tma_prefetch_desc(&kcmap); tma_prefetch_desc(&vcmap); }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  griddep_wait();                         // inputs of earlier stream work are visible
  if (threadIdx.x == 0) *skip_flag = (*(volatile uint32_t*)p.status & kDevTimeout) ? 1u : 0u;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (*skip_flag) {                       // another block already gave up
    if (warp == 1) tmem_dealloc(tmem, 512);
    return;
  }
  const Waiter W{abort_flag, p.status, p.wait_ns};
  // register budgets per warpgroup: warps 0..3 control, 4..11 softmax, 12..15
  // epilogue. The softmax warpgroups' request is the only increase and is met
  // by the two decreases; no warpgroup hands registers back before it exits
  // (an idle control warp doing so early could take them from the pool ahead
  // of the softmax request and stall it).
  if (warp < 4) {
    regs_dec<RegSplit<kSplit>::kCtl>();
    if (warp == 0) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        int gk = 0, lu = 0, q_issued = 0, k_issued = 0, v_issued = 0;
        bool ok = true;
        for (int kk = 0; ok && kk * (int)gridDim.x < total; ++kk) {
          const int u = unit_at(p, kk);
          if (u < 0) continue;
          const WorkItem un = p.units[u / n_hg];
          const int h0 = (u % n_hg) * nh, g = h0 / p.group;
          // Q of this unit once the previous unit's S products are done with it
          if (lu > 0 && !(ok = wait<true>(bar(bQE), (lu - 1) & 1, W, 0x80))) break;
          mbar_arrive_expect_tx(bar(bQF), nh * C::kTile);
          for (int t = 0; t < nh; ++t)
            for (int b = 0; b < NB; ++b)
              tma_load_3d(smem_u32(sQ + t * C::kTile + b * C::kBox), &qmap, bar(bQF), b * 64,
                          h0 + t, un.q0 - p.qbase);
          q_issued = lu + 1;
          for (int it = 0; it < un.nk; ++it) {
            const int gi = gk + it;
            const int32_t c0 = (int32_t)(p.klist[un.kofs + it] & ~kNeedMask);
            // key rows below qbase are cache rows (cached-prefix plans only)
            const bool from_cache = c0 < p.qbase;
            const CUtensorMap* km = from_cache ? &kcmap : &kmap;
            const CUtensorMap* vm = from_cache ? &vcmap : &vmap;
            const int32_t kr = from_cache ? c0 : c0 - p.qbase;
            const int sk = gi % KS, sv = gi % VS;
            if (gi >= KS && !(ok = wait<true>(bar(bKE + sk), ((gi / KS) - 1) & 1, W, 0x100))) break;
            mbar_arrive_expect_tx(bar(bKF + sk), C::kTile);
            for (int b = 0; b < NB; ++b)
              tma_load_3d(smem_u32(sK + sk * C::kTile + b * C::kBox), km, bar(bKF + sk), b * 64,
                          g, kr);
            k_issued = gi + 1;
            if (gi >= VS && !(ok = wait<true>(bar(bVE + sv), ((gi / VS) - 1) & 1, W, 0x180))) break;
            mbar_arrive_expect_tx(bar(bVF + sv), C::kTile);
            for (int b = 0; b < NB; ++b)
              tma_load_3d(smem_u32(sV + sv * C::kTile + b * C::kBox), vm, bar(bVF + sv), b * 64,
                          g, kr);
            v_issued = gi + 1;
          }
          gk += un.nk;
          ++lu;
        }
        // drain: every copy this thread started has landed before the block exits
        if (q_issued > 0) wait_drain(bar(bQF), (q_issued - 1) & 1);
        for (int i = (k_issued > KS ? k_issued - KS : 0); i < k_issued; ++i)
          wait_drain(bar(bKF + i % KS), (i / KS) & 1);
        for (int i = (v_issued > VS ? v_issued - VS : 0); i < v_issued; ++i)
          wait_drain(bar(bVF + i % VS), (i / VS) & 1);
      }
    } else if (warp == 1) {
      // ----------------------------------------------------------------- MMA
      if (lane == 0) {
        constexpr uint32_t idS = idesc_bf16(128, kBN, false);
        constexpr uint32_t idO = idesc_bf16(128, D, true);
        bool ok = true;
        if (p.stall) ok = wait<true>(bar(bDR), 0, W, 0x7ff);   // nothing arrives before the drain
        // S_t = Q_q K^T into the S columns of stream t (q: the Q slot)
        auto issue_s = [&](int t, int q, int sk) {
          const uint32_t aQ = smem_u32(sQ + q * C::kTile);
          const uint32_t aK = smem_u32(sK + sk * C::kTile);
#pragma unroll
          for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_ss(tmem + colS(t), sdesc_sw128(aQ + b * C::kBox + ks * 32, 16, 1024),
                     sdesc_sw128(aK + b * C::kBox + ks * 32, 16, 1024), idS, (b | ks) != 0);
          mma_commit(bar(bSF + t));
        };
        auto issue_pv = [&](int t, int sv, bool acc) {
          const uint32_t aV = smem_u32(sV + sv * C::kTile);
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            // V is MN-major (head dim contiguous): 8-key groups 1024 B apart,
            // 64-column boxes kBox apart. P_t sits in the first columns of S_t.
            const uint64_t db = sdesc_sw128(aV + ks * 16 * 128, C::kBox, 1024);
            mma_ts(tmem + colO(t), tmem + colS(t) + ks * 8, db, idO, (acc || ks != 0) ? 1u : 0u);
          }
        };
        // c0, c1: S products issued so far for each stream (the phase of SF_t / PF_t)
        int gk = 0, lu = 0, c0 = 0, c1 = 0;
        for (int kk = 0; ok && kk * (int)gridDim.x < total; ++kk) {
          const int u = unit_at(p, kk);
          if (u < 0) continue;
          const int nk = p.units[u / n_hg].nk;
          // the unit's Q: landed, or landed and rotated by the softmax warps
          if (!(ok = wait<true>(bar(p.rope ? bQR : bQF), lu & 1, W, 0x200))) break;
          // the first PV of stream t in this unit overwrites O_t: the epilogue of
          // the previous unit must have read it out of tensor memory. In the
          // split schedule one barrier covers both accumulators, and stream 0's
          // first PV always comes first.
          auto first_pv = [&](int t) -> bool {
            if (lu == 0 || (split && t == 1)) return true;
            if (!wait<true>(bar(bOE + t), (lu - 1) & 1, W, 0x280 + t)) return false;
            tc_fence_after();
            return true;
          };
          // unit-local key tile of stream t at step s
          const int ns = split ? (nk + 1) / 2 : nk;
          bool pend1 = false;            // stream 1 owes the PV of the previous step
          int pend1_g = 0;               // ... on this key tile (global index)
          bool pend1_acc = false, pend1_first = false;
          auto flush_pv1 = [&]() -> bool {
            const int pend1_v = pend1_g % VS;
            // split: stream 1's V tile is not stream 0's, wait for it here (in
            // the pair schedule PV_0 of the same tile already waited)
            if (split && !wait<true>(bar(bVF + pend1_v), (pend1_g / VS) & 1, W, 0x3c0))
              return false;
            if (!wait<true>(bar(bPF + 1), (c1 - 1) & 1, W, 0x400)) return false;
            tc_fence_after();
            if (pend1_first && !first_pv(1)) return false;
            issue_pv(1, pend1_v, pend1_acc);
            mma_commit(bar(bVE + pend1_v));
            pend1 = false;
            return true;
          };
          for (int st = 0; ok && st < ns; ++st) {
            const int g0 = gk + (split ? 2 * st : st);
            const int sk0 = g0 % KS, sv0 = g0 % VS;
            if (!(ok = wait<true>(bar(bKF + sk0), (g0 / KS) & 1, W, 0x300))) break;
            tc_fence_after();
            issue_s(0, 0, sk0);
            if (split) mma_commit(bar(bKE + sk0));
            if (pend1 && !(ok = flush_pv1())) break;
            const int i1 = split ? 2 * st + 1 : st;
            if (i1 < nk) {
              const int g1 = gk + i1, sk1 = g1 % KS;
              if (split) {
                if (!(ok = wait<true>(bar(bKF + sk1), (g1 / KS) & 1, W, 0x380))) break;
                tc_fence_after();
              }
              issue_s(1, split ? 0 : 1, sk1);
              mma_commit(bar(bKE + sk1));
              ++c1;
              pend1 = true;
              pend1_g = g1;
              pend1_acc = st > 0;
              pend1_first = st == 0;
            }
            if (st == ns - 1) mma_commit(bar(bQE));        // Q of this unit no longer read
            if (!(ok = wait<true>(bar(bVF + sv0), (g0 / VS) & 1, W, 0x480))) break;
            if (!(ok = wait<true>(bar(bPF + 0), c0 & 1, W, 0x500))) break;
            tc_fence_after();
            if (st == 0 && !(ok = first_pv(0))) break;
            issue_pv(0, sv0, st > 0);
            ++c0;
            if (split) mma_commit(bar(bVE + sv0));
          }
          if (ok && pend1) ok = flush_pv1();
          if (ok) mma_commit(bar(bOF));                    // every PV of the unit done
          gk += nk;
          ++lu;
        }
        // drain: all tensor-core work of this thread completes before dealloc
        mma_commit(bar(bDR));
        wait_drain(bar(bDR), 0);
      }
    }
  } else if (warp < 12) {
    // -------------------------------------------------------------- softmax
    regs_inc<RegSplit<kSplit>::kSoftmax>();
    const int t = (warp - 4) / 4;                       // stream
    const int sw = warp & 3;
    const int r = sw * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(sw * 32) << 16);
    const uint32_t tS = tl + colS(t), tO = tl + colO(t);
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(__float_as_uint(sl2), __float_as_uint(sl2));
    int lu = 0, cs = 0;                                 // cs: S tiles of this stream so far
    bool ok = true;
    for (int kk = 0; ok && kk * (int)gridDim.x < total; ++kk) {
      const int u = unit_at(p, kk);
      if (u < 0) continue;
      const WorkItem un = p.units[u / n_hg];
      const ReqInfo R = p.req[un.req];
      const int j = un.q0 + r;
      const bool valid = j < R.e0;
      const int jj = valid ? j : -1;                    // invalid rows see nothing
      const int lo = valid ? p.seg_start[j - p.qbase] : 0x7fffffff;
      const int nk = un.nk;
      if (p.rope) {
        // rotary embedding of this unit's Q on load, then the MMA thread may
        // read it. Pair schedule: stream t's warps turn rows [64t, 64t + 64)
        // of both heads (16 rows a warp); split schedule: stream t's warps
        // turn half the frequencies of all 128 rows of the one head. Either
        // way every angle is computed once. Positions are the reused ids of
        // Section 4.1 of "From Generation to Scoring": rows of the shared set
        // count from 0 at the request's first row, row d of an item set sits
        // at S + d. Their sines and cosines are computed while the tiles land.
        constexpr int ROWS = split ? 32 : 16;
        const int rr0 = split ? sw * 32 : 64 * t + 16 * sw;
        const int jr = un.q0 + rr0 + lane % ROWS;
        int pos = -1;
        if (jr < R.e0) {
          const int lor = split ? lo : p.seg_start[jr - p.qbase];
          pos = jr < R.pend ? jr - R.s0 : (R.pend - R.s0) + (jr - lor);
        }
        RopeWarp<D, split ? 2 : 1, split ? 1 : 2, ROWS> rw;
        rw.angles(p.rope_freq, pos, split ? t : 0);
        ok = wait<true>(bar(bQF), lu & 1, W, 0x5c0 + t);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        rw.turn(smem_u32(sQ), rr0, split ? t : 0);
        fence_proxy_async();            // the tensor core reads what this warp wrote
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bQR));
      }
      // key tiles of this stream: all (pair) or t, t+2, ... (split)
      const int kstep = split ? 2 : 1, kfirst = split ? t : 0;
      const int nkt = split ? (nk - t + 1) / 2 : nk;
      float m_ref = -INFINITY, l = 0.f;
      uint32_t e_next = nkt > 0 ? p.klist[un.kofs + kfirst] : 0u;
      for (int it = 0; it < nkt; ++it) {
        const int gi = cs + it;
        const uint32_t e = e_next;
        if (it + 1 < nkt) e_next = p.klist[un.kofs + kfirst + (it + 1) * kstep];   // prefetch
        const int32_t c0 = (int32_t)(e & ~kNeedMask);
        const bool masked = (e & kNeedMask) != 0;
        ok = wait<true>(bar(bSF + t), gi & 1, W, 0x600);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        // the whole S row in registers: one load round trip per tile
        uint32_t su[kBN];
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) tmem_ld32(tS + c * 32, su + c * 32);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c) reg_fence32(su + c * 32);
        if (masked) {
          // visible columns of this row: [0, min(row, pend-1) - c0] of the shared
          // set and [lo - c0, row - c0] of its own set, as 4 words of bits
          const int a1 = jj - c0 + 1, q1 = min(a1, R.pend - c0), lc = lo - c0;
#pragma unroll
          for (int w = 0; w < kBN / 32; ++w) {
            const uint32_t vis = bit_range(-32 * w, q1 - 32 * w) | bit_range(lc - 32 * w, a1 - 32 * w);
#pragma unroll
            for (int x = 0; x < 32; ++x)
              if (!((vis >> x) & 1u)) su[w * 32 + x] = 0xff800000u;     // -inf
          }
        }
        // row max: three-input max, four independent chains
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kBN; c += 2)
          mx4[(c >> 1) & 3] = max3(mx4[(c >> 1) & 3], __uint_as_float(su[c]), __uint_as_float(su[c + 1]));
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        const float m_new = fmaxf(m_ref, mx * sl2);
        const bool grow = m_new > m_ref + kRescaleThreshold;
        const bool any_grow = __any_sync(0xffffffffu, grow);
        const float alpha = grow ? ex2(m_ref - m_new) : 1.f;
        if (grow) { l *= alpha; m_ref = m_new; }
        const float mb = (m_ref == -INFINITY) ? 0.f : m_ref;
        // P = 2^(s*scale*log2e - m) as bf16 pairs over the first half of S_h;
        // scale/shift and the row sum run on packed fp32 pairs
        const uint64_t nmbx2 = f2_pack(__float_as_uint(-mb), __float_as_uint(-mb));
        uint64_t rs4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int hf = 0; hf < kBN / 64; ++hf) {        // 64 columns -> 32 packed words
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int k2 = hf * 64 + 2 * c;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(su[k2], su[k2 + 1]), sl2x2, nmbx2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            rs4[c & 3] = f2_add(rs4[c & 3], f2_pack(__float_as_uint(p0), __float_as_uint(p1)));
            pk[c] = pack_bf16(p0, p1);
          }
          tmem_st32(tS + hf * 32, pk);
        }
        {
          float a0, a1;
          f2_unpack(f2_add(f2_add(rs4[0], rs4[1]), f2_add(rs4[2], rs4[3])), a0, a1);
          l += a0 + a1;
        }
        if (any_grow && it > 0) {
          // O_h holds the products up to tile it-1, all complete (see above);
          // it is rescaled after P so that O and S are never live together
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(tO + c * 32, ov);
            tmem_ld_wait();
            reg_fence32(ov);
#pragma unroll
            for (int x = 0; x < 32; ++x) ov[x] = __float_as_uint(__uint_as_float(ov[x]) * alpha);
            tmem_st32(tO + c * 32, ov);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(bPF + t));       // one arrival per warp
      }
      if (!ok) break;
      cs += nkt;
      // hand the row's (max, sum) to the epilogue and go on to the next unit.
      // Slot lu & 1 last held unit lu - 2, which the epilogue has read once
      // SE of the slot completed for it.
      const int slot = lu & 1;
      if (lu >= 2) {
        ok = wait<true>(bar(bSE + slot), ((lu >> 1) - 1) & 1, W, 0x6c0 + t);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      stats[(slot * 2 + t) * kBM + r] = make_float2(m_ref, l);
      mbar_arrive(bar(bST + slot * 2 + t));
      ++lu;
    }
  } else {
    // ------------------------------------------------------------- epilogue
    regs_dec<RegSplit<kSplit>::kEpi>();
    const int sw = warp & 3;
    const int r = sw * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(sw * 32) << 16);
    const uint32_t sOw = smem_u32(sO + sw * C::kOWarp);
    int lu = 0;
    bool ok = true;
    for (int kk = 0; ok && kk * (int)gridDim.x < total; ++kk) {
      const int u = unit_at(p, kk);
      if (u < 0) continue;
      const WorkItem un = p.units[u / n_hg];
      const ReqInfo R = p.req[un.req];
      const int j = un.q0 + r;
      const bool valid = j < R.e0;
      // both streams' (max, sum) of the row; the slot is free once read
      const int slot = lu & 1;
      ok = wait<true>(bar(bST + slot * 2), (lu >> 1) & 1, W, 0x700) &&
           wait<true>(bar(bST + slot * 2 + 1), (lu >> 1) & 1, W, 0x701);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const float2 s0 = stats[(slot * 2) * kBM + r], s1 = stats[(slot * 2 + 1) * kBM + r];
      mbar_arrive(bar(bSE + slot));
      ok = wait<true>(bar(bOF), lu & 1, W, 0x740);          // every PV of the unit done
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // O leaves through a 32-row x 64-column staging buffer per warp and a
      // TMA tensor store (asynchronous, whole rows); a warp whose 32 rows run
      // past the request's end stores its valid rows directly instead, since
      // the rows after them belong to the next request
      const int row0 = un.q0 + sw * 32;
      const bool wfull = row0 + 32 <= R.e0;
      auto stage_begin = [&]() {                        // the previous store has read the buffer
        if (lane == 0) bulk_wait_read0();
        __syncwarp();
      };
      // 32 columns (16 bf16 pairs) of this row: piece q of the staged 64 columns
      auto stage16 = [&](const uint32_t* pk, int q) {
        const uint32_t ra = sOw + lane * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {                   // 128-byte swizzle: chunk cc ^ (row & 7)
          const int cc = q * 4 + c;
          st_shared_v4(ra + ((cc ^ (lane & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                       pk[4 * c + 3]);
        }
      };
      auto stage_end = [&](int col0, int h) {
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&omap, sOw, col0, h, row0 - p.qbase);
          bulk_commit();
        }
      };
      // 16 columns (8 bf16 pairs): piece q of the staged 64 columns
      auto stage8 = [&](const uint32_t* pk, int q) {
        const uint32_t ra = sOw + lane * 128;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int cc = q * 2 + c;
          st_shared_v4(ra + ((cc ^ (lane & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                       pk[4 * c + 3]);
        }
      };
      auto direct8 = [&](const uint32_t* pk, int col0, int h) {
        if (!valid) return;
        uint4* dst = reinterpret_cast<uint4*>(p.o + (int64_t)(j - p.qbase) * p.o_stride +
                                              (int64_t)h * D + col0);
        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      };
      auto direct16 = [&](const uint32_t* pk, int col0, int h) {
        if (!valid) return;
        uint4* dst = reinterpret_cast<uint4*>(p.o + (int64_t)(j - p.qbase) * p.o_stride +
                                              (int64_t)h * D + col0);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      };
      if (!split) {
        // head t of the pair: O_t / l_t, 32 columns at a time; O_t goes back
        // to the MMA thread as soon as its last columns are read
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float2 st = t == 0 ? s0 : s1;
          const int h = (u % n_hg) * 2 + t;
          const float inv = st.y > 0.f ? 1.f / st.y : 0.f;
          const uint32_t tO = tl + colO(t);
#pragma unroll
          for (int hh = 0; hh < D / 64; ++hh) {
            if (wfull) stage_begin();
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              uint32_t ov[32];
              tmem_ld32(tO + hh * 64 + q * 32, ov);
              tmem_ld_wait();
              reg_fence32(ov);
              if (hh == D / 64 - 1 && q == 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(bOE + t));
              }
              uint32_t pk[16];
#pragma unroll
              for (int x = 0; x < 16; ++x)
                pk[x] = pack_bf16(__uint_as_float(ov[2 * x]) * inv,
                                  __uint_as_float(ov[2 * x + 1]) * inv);
              if (wfull) stage16(pk, q);
              else direct16(pk, hh * 64 + q * 32, h);
            }
            if (wfull) stage_end(hh * 64, h);
          }
          if (p.lse && valid) p.lse[(int64_t)h * p.T + (j - p.qbase)] = (st.x + log2f(st.y)) * kLn2;
        }
      } else {
        // merge the two streams' partial results of this row:
        //   m = max(m_0, m_1), a_s = 2^(m_s - m), L = a_0 l_0 + a_1 l_1,
        //   O = (a_0 O_0 + a_1 O_1) / L.
        const int h = u % n_hg;
        const float m = fmaxf(s0.x, s1.x);
        const float a0 = (m == -INFINITY) ? 0.f : ex2(s0.x - m);
        const float a1 = (m == -INFINITY) ? 0.f : ex2(s1.x - m);
        const float L = s0.y * a0 + s1.y * a1;
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const float w0 = a0 * inv, w1 = a1 * inv;
        const bool has1 = un.nk > 1;                    // stream 1 wrote O_1 in this unit
        const uint32_t tO0 = tl + colO(0), tO1 = tl + colO(1);
#pragma unroll
        for (int hh = 0; hh < D / 64; ++hh) {
          if (wfull) stage_begin();
#pragma unroll
          for (int q = 0; q < 4; ++q) {                 // 16 columns of each accumulator at a time
            const int c = hh * 64 + q * 16;
            // O_1 is read even when stream 1 had no tile (then it holds an
            // older unit's values, or nothing ever written) and dropped by a
            // select
            uint32_t o0[16], o1[16];
            tmem_ld16(tO0 + c, o0);
            tmem_ld16(tO1 + c, o1);
            tmem_ld_wait();
            reg_fence16(o0);
            reg_fence16(o1);
            if (hh == D / 64 - 1 && q == 3) {           // both accumulators read: hand them back
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar(bOE + 0));
            }
            uint32_t pk[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
              float v2[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const float a = __uint_as_float(o0[2 * x + e]) * w0;
                v2[e] = has1 ? fmaf(__uint_as_float(o1[2 * x + e]), w1, a) : a;
              }
              pk[x] = pack_bf16(v2[0], v2[1]);
            }
            if (wfull) stage8(pk, q);
            else direct8(pk, c, h);
          }
          if (wfull) stage_end(hh * 64, h);
        }
        if (p.lse && valid) p.lse[(int64_t)h * p.T + (j - p.qbase)] = (m + log2f(L)) * kLn2;
      }
      ++lu;
    }
    if (lane == 0) bulk_wait0();          // O stores complete before the block exits
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
mis_status_t launch_d(HostPlan& pl, const void* q, const void* k, const void* v,
                      const void* kc, const void* vc, void* o, float* lse, int64_t qs, int64_t ks,
                      int64_t vs, int64_t kcs, int64_t vcs, int64_t os, const RopeQ* rope,
                      void* stream) {
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
  const uint32_t obox[3] = {64, 1, 32};
  const uint64_t ostr[2] = {(uint64_t)D * 2, (uint64_t)os * 2};
  CUtensorMap om = make_tmap_bf16(o, 3, qd, ostr, obox, &ok);
  CUtensorMap kcm = km, vcm = vm;
  if (pl.cached) {
    const uint64_t cd[3] = {(uint64_t)D, (uint64_t)pl.Hkv, (uint64_t)pl.cache_T};
    const uint64_t kcstr[2] = {(uint64_t)D * 2, (uint64_t)kcs * 2};
    const uint64_t vcstr[2] = {(uint64_t)D * 2, (uint64_t)vcs * 2};
    kcm = make_tmap_bf16(kc, 3, cd, kcstr, box, &ok);
    vcm = make_tmap_bf16(vc, 3, cd, vcstr, box, &ok);
  }
  if (!ok) return MIS_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(pl.workspace);
  AttnParams prm;
  prm.req = reinterpret_cast<const ReqInfo*>(ws + pl.off_req);
  prm.seg_start = reinterpret_cast<const int32_t*>(ws + pl.off_seg);
  prm.units = reinterpret_cast<const WorkItem*>(ws + pl.off_work);
  prm.klist = reinterpret_cast<const uint32_t*>(ws + pl.off_klist);
  prm.n_units = (int32_t)pl.work.size();
  prm.order = pl.order.empty() ? nullptr : reinterpret_cast<const int32_t*>(ws + pl.off_order);
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.o_stride = os;
  prm.T = pl.T;
  prm.qbase = pl.cached ? pl.qbase : 0;
  prm.group = pl.Hq / pl.Hkv;
  prm.n_head_groups = pl.n_head_groups;
  prm.scale_log2 = pl.scale * 1.4426950408889634f;
  prm.status = reinterpret_cast<uint32_t*>(ws);
  prm.wait_ns = wait_limit_ns();
  prm.stall = inject_stall_mask() & 1u;
  prm.rope = rope ? 1 : 0;
  for (int i = 0; i < 64; ++i)
    prm.rope_freq[i] = (rope && i < D / 2) ? (float)std::pow(rope->base, -2.0 * i / D) : 0.f;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (pl.status_clear) {
    pl.status_clear = false;               // zeroed by the plan upload just before
  } else if (cudaMemsetAsync(ws, 0, 8, st) != cudaSuccess) {
    return MIS_ERR_CUDA;
  }
  if (pl.work.empty()) return MIS_OK;
  auto kern = pl.split ? mis_attn_fwd_kernel<D, true> : mis_attn_fwd_kernel<D, false>;
  if (!kernel_attr_once(reinterpret_cast<const void*>(kern), C::kSmem)) return MIS_ERR_CUDA;
  const int64_t total = (int64_t)pl.work.size() * pl.n_head_groups;
  if (total > 0x7fffffff) return MIS_ERR_UNSUPPORTED;
  prm.n_walk = pl.order.empty() ? (int32_t)total : (int32_t)pl.order.size();
  dim3 grid((unsigned)std::min<int64_t>(total, num_sms()));
  return launch_pdl(kern, grid, dim3(kThreads), C::kSmem, st, qm, km, vm, om, kcm, vcm, prm) ==
                 cudaSuccess
             ? MIS_OK
             : MIS_ERR_CUDA;
}

}  // namespace

mis_status_t launch_attention(HostPlan& p, const void* q, const void* k, const void* v,
                              const void* k_cache, const void* v_cache, void* o, float* lse,
                              int64_t qs, int64_t ks, int64_t vs, int64_t kcs, int64_t vcs,
                              int64_t os, void* stream, const RopeQ* rope) {
  if (p.D == 128)
    return launch_d<128>(p, q, k, v, k_cache, v_cache, o, lse, qs, ks, vs, kcs, vcs, os, rope,
                         stream);
  if (p.D == 64)
    return launch_d<64>(p, q, k, v, k_cache, v_cache, o, lse, qs, ks, vs, kcs, vcs, os, rope,
                        stream);
  return MIS_ERR_UNSUPPORTED;
}

}  // namespace mis
