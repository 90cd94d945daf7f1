// Label scoring at the MIS readout rows, sm_103a.
//
// For every item i with readout row r_i (its trailing DELIM):
//   z_i = W_lm h_{r_i}  over the whole vocabulary,
//   logprob[i, l] = z_i[label_l] - logsumexp_v z_i[v],
//   renorm[i, :]  = softmax over the K label logits (eq. 2 for K = 2).
// ("From Generation to Scoring: Scaling LLM-Based Semantic Labeling at
// LinkedIn", Section 3.3; "Scaling JEV-like Decision Models with SGLang",
// "Why a Decision Workload Deserves a Scoring Interface": label extraction
// keeps the vocabulary projection and the full-distribution normalisation;
// "Turbocharging LinkedIn's recommendation systems with SGLang", "SGLang
// changes": an N x K matrix of label log-probs.)
//
// Three launches:
//   1. gather  — copy the M readout rows of `hidden` into a dense [M_pad, d]
//                bf16 block (M_pad a multiple of 128, zero rows after M);
//   2. partial — grid (item tile, vocab chunk). Each block multiplies one
//                128-item tile against a run of 256-token vocab tiles on the
//                tensor cores (tcgen05.mma 128x256x16, both operands staged by
//                TMA with 128-byte swizzle, fp32 accumulators in TMEM, two
//                accumulators so the epilogue of tile t overlaps the MMAs of
//                tile t+1). The epilogue reads each item's 256 logits from its
//                TMEM lane, folds them into a running (max, sum of exp) and
//                keeps the logits of requested labels. Logits never reach
//                global memory; only one (max, sum) pair per item and chunk;
//   3. combine — merge the pairs of all chunks into logsumexp, write the
//                label log-probs and the label-renormalised scores.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "mis_internal.h"
#include "mis_ptx.cuh"

namespace mis {

CUtensorMap make_tmap_bf16(const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box, bool* ok);

namespace {

using namespace dev;

constexpr int kItemTile = 128;   // MMA M: items
constexpr int kVocabTile = 256;  // MMA N: vocabulary entries
constexpr int kKStep = 64;       // d elements per stage (one 128-byte swizzle row)
constexpr int kStages = 4;
constexpr int kABytes = kItemTile * kKStep * 2;    // 16 KB
constexpr int kBBytes = kVocabTile * kKStep * 2;   // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kData = kStages * kStageBytes;
constexpr int kSmem = kData + 256 + 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994530942f;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct ScoreLayout {       // byte offsets inside the scoring workspace
  size_t gathered, part, zlab, bad, total;
  int32_t m_pad, n_vtiles, max_chunks;
};

ScoreLayout score_layout(int32_t M, int32_t d, int32_t V, int32_t K) {
  ScoreLayout L;
  // several item tiles run on CTA pairs (one 256-row product over two SMs):
  // an even number of them
  L.m_pad = M <= kItemTile ? kItemTile : (int32_t)align_up((size_t)M, 2 * kItemTile);
  L.n_vtiles = (V + kVocabTile - 1) / kVocabTile;
  L.max_chunks = L.n_vtiles;
  size_t off = kStatusBytes;
  L.gathered = off; off = align_up(off + (size_t)L.m_pad * d * 2, 1024);
  L.part = off;     off = align_up(off + (size_t)L.m_pad * L.max_chunks * 2 * sizeof(float), 256);
  L.zlab = off;     off = align_up(off + (size_t)L.m_pad * std::max(K, 1) * sizeof(float), 256);
  L.bad = off;      off = align_up(off + (size_t)L.m_pad * sizeof(int32_t), 256);
  L.total = off;
  return L;
}

struct ScoreParams {
  int32_t M, V, K, n_vtiles, tiles_per_chunk, n_chunks, n_kb;
  int32_t n_parts;         // (max, sum) partials per item: one per chunk, or one per vocabulary
                           // tile when the tiles come from the counter (a fixed merge order, so
                           // the scores repeat bit for bit whichever block ran which tile)
  int32_t dynamic;         // one item tile: blocks take vocabulary tiles from a counter
  uint32_t* ctr;           // that counter (a status word, cleared by the gather kernel)
  const uint8_t* w_lm;     // W_lm rows, for the L2 prefetch
  uint32_t pf_bytes;       // W_lm bytes of its range each block prefetches into L2 before its wait
  int32_t labels[16];
  float* part;        // [m_pad][n_parts][2] = (max in log2 units, sum of 2^(z*log2e - max))
  float* zlab;        // [m_pad][K] label logits
  const int32_t* bad; // [m_pad] 1 where the readout row was out of range
  uint32_t* status;
  uint64_t wait_ns;
  uint32_t stall;     // failure injection: wait on a barrier nothing arrives on
};

// ------------------------------------------------------------------ gather
// Also starts the call's device status: block 0 clears the status words (no
// other block of this launch writes them; an out-of-range row is recorded in
// bad[] and raised by the combine kernel, which runs after every block here).
// It lets the LM-head kernel launch at once, before its own wait: the LM-head
// kernel reads only W_lm before its griddepcontrol.wait, which waits for this
// grid and so for everything before it.
__global__ void __launch_bounds__(128)
mis_gather_rows_kernel(const __nv_bfloat16* __restrict__ hidden, int64_t stride, int32_t T,
                       const int32_t* __restrict__ rows, int32_t M, int32_t d,
                       __nv_bfloat16* __restrict__ out, int32_t* __restrict__ bad,
                       uint32_t* status) {
  griddep_launch_dependents();
  griddep_wait();
  const int i = blockIdx.x;
  if (i == 0 && threadIdx.x == 0) {
    status[0] = 0u;
    status[1] = 0u;
    status[2] = 0u;                                   // the LM head's vocabulary-tile counter
  }
  int32_t r = -1;
  if (i < M) {
    r = rows[i];
    if (r < 0 || r >= T) r = -1;
  }
  if (threadIdx.x == 0) bad[i] = (i < M && r < 0) ? 1 : 0;
  const int n16 = d / 8;                              // 16-byte chunks per row
  uint4* dst = reinterpret_cast<uint4*>(out + (int64_t)i * d);
  if (r < 0) {
    for (int c = threadIdx.x; c < n16; c += blockDim.x) dst[c] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(hidden + (int64_t)r * stride);
  for (int c = threadIdx.x; c < n16; c += blockDim.x) dst[c] = src[c];
}

// ----------------------------------------------------------------- partial
// Vocabulary tiles per block: a fixed run of tiles_per_chunk tiles (grid
// (item tiles, chunks)), or, with one item tile, tiles taken from a global
// counter (grid (1, G), G <= SMs): block b starts with tile b and then takes
// G + counter++ until the tiles run out, so blocks that stream faster take
// more tiles and all finish together. The producer hands each tile index to
// the MMA thread and the epilogue warps through a ring in shared memory
// (index -1 ends the block's work).
constexpr int kRing = 4;

__global__ void __launch_bounds__(256, 1)
mis_score_partial_kernel(const __grid_constant__ CUtensorMap amap,
                         const __grid_constant__ CUtensorMap wmap, const ScoreParams p) {
  griddep_launch_dependents();
  constexpr int bF = 0, bE = kStages, bAF = 2 * kStages, bAE = bAF + 2, bDR = bAE + 2,
                bTF = bDR + 1, bTE = bTF + kRing, nBar = bTE + kRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kData);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + nBar);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* skip_flag = tmem_slot + 2;
  volatile int32_t* ring = reinterpret_cast<volatile int32_t*>(tmem_slot + 4);   // kRing entries
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = blockIdx.x;
  const int chunk = blockIdx.y;
  const bool dyn = p.dynamic != 0;
  const int G = (int)gridDim.y;
  const int v_first = dyn ? chunk : chunk * p.tiles_per_chunk;   // the block's first tile
  const int v_last = dyn ? p.n_vtiles : min(v_first + p.tiles_per_chunk, p.n_vtiles);
  const bool has_work = v_first < v_last;
  const int nkb = p.n_kb;

  // prologue (shared memory and tensor memory only) overlaps the previous
  // kernel in the stream; global memory other than W_lm is read after
  // griddepcontrol.wait
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStages; ++s) { mbar_init(bar(bF + s), 1); mbar_init(bar(bE + s), 1); }
    for (int s = 0; s < 2; ++s) { mbar_init(bar(bAF + s), 1); mbar_init(bar(bAE + s), 128); }
    mbar_init(bar(bDR), 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(bar(bTF + s), 1);
      mbar_init(bar(bTE + s), 5);                       // the MMA thread and 4 epilogue warps
    }
    fence_mbar_init();
    fence_proxy_async();
  }
  // W_lm is a weight: the stream work before this call does not write it (a
  // documented rule of mis_label_scores), so it is read before
  // griddepcontrol.wait. The gather kernel lets this grid launch as soon as
  // its blocks start, so blocks start here while the kernels before the call
  // (e.g. the attention layer) drain: the first stages of the block's first
  // W_lm tile load into shared memory and the next part of that tile into L2
  // while HBM is otherwise idle. Only the readout-row tiles wait for the
  // gather.
  const int pre = has_work ? min(kStages, nkb) : 0;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&amap);
    tma_prefetch_desc(&wmap);
    for (int step = 0; step < pre; ++step) {
      mbar_expect_tx(bar(bF + step), kBBytes);
      tma_load_2d(smem_u32(smem + step * kStageBytes + kABytes), &wmap, bar(bF + step),
                  step * kKStep, v_first * kVocabTile);
    }
    if (p.pf_bytes && has_work && blockIdx.x == 0) {
      // the rows of a run of tiles are one contiguous range of W_lm
      const size_t row_bytes = (size_t)nkb * kKStep * 2;
      const size_t v0 = (size_t)v_first * kVocabTile;
      const size_t v1 = min((size_t)(dyn ? v_first + 1 : v_last) * kVocabTile, (size_t)p.V);
      const size_t range = (v1 - v0) * row_bytes;
      const uint8_t* base = p.w_lm + v0 * row_bytes;
      const size_t n = min((size_t)p.pf_bytes, range) & ~(size_t)15;
      for (size_t off = 0; off < n; off += 65536)
        bulk_prefetch_l2(base + off, (uint32_t)min((size_t)65536, n - off));
    }
  }
  if (warp == 1 && has_work) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  griddep_wait();
  if (threadIdx.x == 0) *skip_flag = (*(volatile uint32_t*)p.status & kDevTimeout) ? 1u : 0u;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!has_work) return;
  const uint32_t tmem = *tmem_slot;
  if (*skip_flag) {                       // another block already gave up
    if (threadIdx.x == 0)                 // the early W_lm copies land before the block exits
      for (int step = 0; step < pre; ++step) {
        mbar_arrive(bar(bF + step));
        wait_drain(bar(bF + step), 0);
      }
    if (warp == 1) tmem_dealloc(tmem, 512);
    return;
  }
  const Waiter W{abort_flag, p.status, p.wait_ns};

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0, step = 0;
      int t = v_first;
      // the tile after the current one, asked for one tile ahead (the
      // counter's round trip hides behind the current tile's loads)
      int t_next = dyn ? G + (int)atomicAdd(p.ctr, 1u) : v_first + 1;
      for (int j = 0;; ++j) {
        const int slot = j % kRing;
        if (j >= kRing && !wait(bar(bTE + slot), ((j / kRing) - 1) & 1, W, 0x080)) break;
        const bool valid = t < v_last;
        ring[slot] = valid ? t : -1;
        mbar_arrive(bar(bTF + slot));
        if (!valid) break;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++step) {
          const int st = step % kStages;
          if (step >= kStages && !wait(bar(bE + st), ((step / kStages) - 1) & 1, W, 0x100)) {
            ok = false;
            break;
          }
          uint8_t* sA = smem + st * kStageBytes;
          uint8_t* sB = sA + kABytes;
          if (step < pre) {               // W_lm tile already on its way
            mbar_arrive_expect_tx(bar(bF + st), kABytes);
            tma_load_2d(smem_u32(sA), &amap, bar(bF + st), kb * kKStep, mt * kItemTile);
          } else {
            mbar_arrive_expect_tx(bar(bF + st), kStageBytes);
            tma_load_2d(smem_u32(sA), &amap, bar(bF + st), kb * kKStep, mt * kItemTile);
            tma_load_2d(smem_u32(sB), &wmap, bar(bF + st), kb * kKStep, t * kVocabTile);
          }
          issued = step + 1;
        }
        if (!ok) break;
        t = t_next;
        if (t < v_last) t_next = dyn ? G + (int)atomicAdd(p.ctr, 1u) : t + 1;
      }
      for (int i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
        wait_drain(bar(bF + i % kStages), (i / kStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kItemTile, kVocabTile, false);
      bool ok = true;
      if (p.stall) ok = wait(bar(bDR), 0, W, 0x7ff);   // nothing arrives before the drain
      for (int j = 0; ok; ++j) {
        const int slot = j % kRing;
        if (!wait(bar(bTF + slot), (j / kRing) & 1, W, 0x180)) break;
        const int t = ring[slot];
        mbar_arrive(bar(bTE + slot));
        if (t < 0) break;
        const int buf = j & 1;
        if (j >= 2 && !wait(bar(bAE + buf), ((j >> 1) - 1) & 1, W, 0x200)) break;
        tc_fence_after();
        const uint32_t dacc = tmem + buf * kVocabTile;
        for (int kb = 0; kb < nkb; ++kb) {
          const int step = j * nkb + kb;
          const int st = step % kStages;
          if (!wait(bar(bF + st), (step / kStages) & 1, W, 0x300)) { ok = false; break; }
          tc_fence_after();
          const uint32_t aA = smem_u32(smem + st * kStageBytes);
          const uint32_t aB = aA + kABytes;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ss(dacc, sdesc_sw128(aA + ks * 32, 16, 1024), sdesc_sw128(aB + ks * 32, 16, 1024),
                   idesc, (kb | ks) != 0);
          mma_commit(bar(bE + st));
        }
        if (ok) mma_commit(bar(bAF + buf));
      }
      mma_commit(bar(bDR));
      wait_drain(bar(bDR), 0);
    }
  } else if (warp >= 4) {
    const int sw = warp - 4;
    const int row = sw * 32 + lane;
    const int item = mt * kItemTile + row;
    const uint32_t tl = tmem + ((uint32_t)(sw * 32) << 16);
    float m2 = -INFINITY, s = 0.f;
    bool ok = true;
    for (int j = 0;; ++j) {
      const int slot = j % kRing;
      ok = wait(bar(bTF + slot), (j / kRing) & 1, W, 0x380);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int t = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bTE + slot));
      if (t < 0) break;
      const int buf = j & 1;
      ok = wait(bar(bAF + buf), (j >> 1) & 1, W, 0x400);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int v0 = t * kVocabTile;
      const uint32_t tacc = tl + buf * kVocabTile;
#pragma unroll 1
      for (int c = 0; c < kVocabTile / 32; ++c) {
        uint32_t zr[32];
        tmem_ld32(tacc + c * 32, zr);
        tmem_ld_wait();
        reg_fence32(zr);
        const int vbase = v0 + c * 32;
        float cm = -INFINITY;
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const float z = (vbase + x < p.V) ? __uint_as_float(zr[x]) * kLog2e : -INFINITY;
          zr[x] = __float_as_uint(z);
          cm = fmaxf(cm, z);
        }
        if (cm > m2) {
          s *= ex2(m2 - cm);
          m2 = cm;
        }
        float cs = 0.f;
#pragma unroll
        for (int x = 0; x < 32; ++x) cs += ex2(__uint_as_float(zr[x]) - m2);
        s += cs;
      }
      for (int l = 0; l < p.K; ++l) {
        const int lab = p.labels[l];
        if (lab >= v0 && lab < v0 + kVocabTile) {
          uint32_t z = tmem_ld1(tacc + (lab - v0));
          tmem_ld_wait();
          reg_fence1(z);
          if (item < p.M) p.zlab[(int64_t)item * p.K + l] = __uint_as_float(z);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(bAE + buf));
      if (dyn) {                                      // this tile's own partial
        float* pp = p.part + ((int64_t)item * p.n_parts + t) * 2;
        pp[0] = m2;
        pp[1] = s;
        m2 = -INFINITY;
        s = 0.f;
      }
    }
    if (ok && !dyn) {
      float* pp = p.part + ((int64_t)item * p.n_parts + chunk) * 2;
      pp[0] = m2;
      pp[1] = s;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------- partial, SM pairs
// The same (item tile, run of vocabulary tiles) work as the kernel above, on
// a cluster of two CTAs on two SMs: item tiles 2i and 2i + 1 (one per CTA)
// against one run of vocabulary tiles. Each 256 x 256 x 16 product is one
// tcgen05.mma.cta_group::2 issued by the even CTA: A rows (items) and the
// accumulator rows stay in their own CTA, and each CTA holds half of the
// W_lm tile (vocabulary rows v0 + 128 r .. v0 + 128 r + 127 in CTA r). Per SM
// the W_lm tile's shared-memory fills and operand reads are half of the
// single-SM kernel's, which ran short of shared-memory bandwidth rather than
// tensor-core rate. Both CTAs' TMA loads of a stage complete on the even
// CTA's full barrier; its MMA thread's commits arrive on the barriers of both
// CTAs; each CTA's epilogue reads its own accumulator rows and releases the
// accumulator with an arrival on the even CTA's barrier.
constexpr int kPairStages = 6;
constexpr int kBHalfBytes = (kVocabTile / 2) * kKStep * 2;   // 16 KB
constexpr int kPairStageBytes = kABytes + kBHalfBytes;
constexpr int kPairData = kPairStages * kPairStageBytes;
constexpr int kPairSmem = kPairData + 512 + 1024;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
mis_score_partial_pair_kernel(const __grid_constant__ CUtensorMap amap,
                              const __grid_constant__ CUtensorMap wmap, const ScoreParams p) {
  griddep_launch_dependents();
  constexpr int S = kPairStages;
  constexpr int bF = 0, bE = S, bAF = 2 * S, bAE = bAF + 2, bDR = bAE + 2, bTF = bDR + 1,
                bTE = bTF + kRing, nBar = bTE + kRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPairData);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + nBar);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile int32_t* ring = reinterpret_cast<volatile int32_t*>(tmem_slot + 4);   // kRing entries
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int mt = blockIdx.x;                      // this CTA's item tile
  const int chunk = blockIdx.y;
  const int v_first = chunk * p.tiles_per_chunk;
  const int v_last = min(v_first + p.tiles_per_chunk, p.n_vtiles);
  const int nkb = p.n_kb;
  // the even CTA's barrier at the offset of this CTA's `i`
  auto lbar = [&](int i) { return mapa_shared(bar(i), 0); };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int st = 0; st < S; ++st) { mbar_init(bar(bF + st), 1); mbar_init(bar(bE + st), 1); }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(bAF + b), 1);
      mbar_init(bar(bAE + b), 8);                     // the epilogue warps of both CTAs
    }
    mbar_init(bar(bDR), 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(bar(bTF + s), 1);
      mbar_init(bar(bTE + s), leader ? 5 : 4);        // (the MMA thread) and 4 epilogue warps
    }
    fence_mbar_init();
    fence_proxy_async();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&amap);
    tma_prefetch_desc(&wmap);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  // both CTAs' barriers are initialised before any arrival or copy crosses
  cluster_sync_all();
  griddep_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{abort_flag, p.status, p.wait_ns};

  if (warp == 0) {
    if (lane == 0) {
      int step = 0;
      for (int j = 0, t = v_first;; ++j, ++t) {
        const int slot = j % kRing;
        if (j >= kRing && !wait(bar(bTE + slot), ((j / kRing) - 1) & 1, W, 0x880)) break;
        const bool valid = t < v_last;
        ring[slot] = valid ? t : -1;
        mbar_arrive(bar(bTF + slot));
        if (!valid) break;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb, ++step) {
          const int st = step % S;
          if (step >= S && !wait(bar(bE + st), ((step / S) - 1) & 1, W, 0x900)) {
            ok = false;
            break;
          }
          // the even CTA's full barrier counts both CTAs' bytes of the stage
          if (leader) mbar_arrive_expect_tx(bar(bF + st), 2 * kPairStageBytes);
          uint8_t* sA = smem + st * kPairStageBytes;
          tma_load_2d_pair(smem_u32(sA), &amap, lbar(bF + st), kb * kKStep, mt * kItemTile);
          tma_load_2d_pair(smem_u32(sA + kABytes), &wmap, lbar(bF + st), kb * kKStep,
                           t * kVocabTile + (int)rank * (kVocabTile / 2));
        }
        if (!ok) break;
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(2 * kItemTile, kVocabTile, false);
      bool ok = true;
      if (p.stall) ok = wait(bar(bDR), 0, W, 0xfff);   // nothing arrives before the drain
      for (int j = 0; ok; ++j) {
        const int slot = j % kRing;
        if (!wait(bar(bTF + slot), (j / kRing) & 1, W, 0x980)) break;
        const int t = ring[slot];
        mbar_arrive(bar(bTE + slot));
        if (t < 0) break;
        const int buf = j & 1;
        if (j >= 2 && !wait_cluster(bar(bAE + buf), ((j >> 1) - 1) & 1, W, 0xa00)) break;
        tc_fence_after();
        const uint32_t dacc = tmem + buf * kVocabTile;
        for (int kb = 0; kb < nkb; ++kb) {
          const int step = j * nkb + kb;
          const int st = step % S;
          if (!wait(bar(bF + st), (step / S) & 1, W, 0xb00)) { ok = false; break; }
          tc_fence_after();
          const uint32_t aA = smem_u32(smem + st * kPairStageBytes);
          const uint32_t aB = aA + kABytes;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ss_pair(dacc, sdesc_sw128(aA + ks * 32, 16, 1024),
                        sdesc_sw128(aB + ks * 32, 16, 1024), idesc, (kb | ks) != 0);
          mma_commit_pair(bar(bE + st), 0x3);         // the stage is free in both CTAs
        }
        if (ok) mma_commit_pair(bar(bAF + buf), 0x3); // the accumulators are complete
      }
      // drain: every product this thread issued has completed, and every copy
      // of a stage it waited for has landed
      mma_commit_pair(bar(bDR), 0x1);
      wait_drain(bar(bDR), 0);
    }
  } else if (warp >= 4) {
    const int sw = warp - 4;
    const int row = sw * 32 + lane;
    const int item = mt * kItemTile + row;
    const uint32_t tl = tmem + ((uint32_t)(sw * 32) << 16);
    float m2 = -INFINITY, s = 0.f;
    bool ok = true;
    for (int j = 0;; ++j) {
      const int slot = j % kRing;
      ok = wait(bar(bTF + slot), (j / kRing) & 1, W, 0xb80);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int t = ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(bTE + slot));
      if (t < 0) break;
      const int buf = j & 1;
      ok = wait(bar(bAF + buf), (j >> 1) & 1, W, 0xc00);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int v0 = t * kVocabTile;
      const uint32_t tacc = tl + buf * kVocabTile;
#pragma unroll 1
      for (int c = 0; c < kVocabTile / 32; ++c) {
        uint32_t zr[32];
        tmem_ld32(tacc + c * 32, zr);
        tmem_ld_wait();
        reg_fence32(zr);
        const int vbase = v0 + c * 32;
        float cm = -INFINITY;
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const float z = (vbase + x < p.V) ? __uint_as_float(zr[x]) * kLog2e : -INFINITY;
          zr[x] = __float_as_uint(z);
          cm = fmaxf(cm, z);
        }
        if (cm > m2) {
          s *= ex2(m2 - cm);
          m2 = cm;
        }
        float cs = 0.f;
#pragma unroll
        for (int x = 0; x < 32; ++x) cs += ex2(__uint_as_float(zr[x]) - m2);
        s += cs;
      }
      for (int l = 0; l < p.K; ++l) {
        const int lab = p.labels[l];
        if (lab >= v0 && lab < v0 + kVocabTile) {
          uint32_t z = tmem_ld1(tacc + (lab - v0));
          tmem_ld_wait();
          reg_fence1(z);
          if (item < p.M) p.zlab[(int64_t)item * p.K + l] = __uint_as_float(z);
        }
      }
      // the accumulator may be overwritten once both CTAs' epilogues read it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(lbar(bAE + buf));
    }
    if (ok) {
      float* pp = p.part + ((int64_t)item * p.n_parts + chunk) * 2;
      pp[0] = m2;
      pp[1] = s;
    }
  }
  // no CTA of the pair leaves (and frees its tensor memory) while the other
  // may still issue products into it or copies onto its barriers
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

// ----------------------------------------------------------------- combine
// One warp per item: lanes stride over the vocab chunks, then merge their
// (max, sum) pairs with shuffles.
__global__ void __launch_bounds__(128)
mis_score_combine_kernel(const ScoreParams p, float* __restrict__ out,
                         float* __restrict__ renorm) {
  griddep_wait();
  griddep_launch_dependents();
  const int i = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= p.M) return;
  if (lane == 0 && p.bad[i]) raise_status(p.status, kDevIndex, (uint32_t)i);
  if (*(volatile uint32_t*)p.status & kDevTimeout) return;
  const float2* pp = reinterpret_cast<const float2*>(p.part) + (int64_t)i * p.n_parts;
  float m = -INFINITY, s = 0.f;
  // up to 24 partials per lane are loaded together, then merged: one L2 round
  // trip per 768 partials (a 151,936-entry vocabulary has 594) instead of one
  // per 32
  constexpr int kPer = 24;
  for (int c0 = lane; c0 < p.n_parts; c0 += 32 * kPer) {
    float2 e[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int c = c0 + 32 * u;
      e[u] = c < p.n_parts ? pp[c] : make_float2(-INFINITY, 0.f);
    }
    // the batch's max first, then its sum: independent exponentials, no
    // chain of dependent rescales
    float mb = -INFINITY;
#pragma unroll
    for (int u = 0; u < kPer; ++u) mb = fmaxf(mb, e[u].x);
    if (mb == -INFINITY) continue;
    float sb = 0.f;
#pragma unroll
    for (int u = 0; u < kPer; ++u) sb += e[u].y * exp2f(e[u].x - mb);    // exp2f(-inf) = 0
    const float mm = fmaxf(m, mb);
    s = (m == -INFINITY ? 0.f : s * exp2f(m - mm)) + sb * exp2f(mb - mm);
    m = mm;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float so = __shfl_xor_sync(0xffffffffu, s, off);
    const float mm = fmaxf(m, mo);
    if (mm != -INFINITY) s = s * exp2f(m - mm) + so * exp2f(mo - mm);
    m = mm;
  }
  const float lse = (m + log2f(s)) * kLn2;
  const float* zl = p.zlab + (int64_t)i * p.K;
  if (lane < p.K) out[(int64_t)i * p.K + lane] = zl[lane] - lse;
  if (renorm) {
    const float z = lane < p.K ? zl[lane] : -INFINITY;
    float zmax = z;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, off));
    float e = lane < p.K ? expf(z - zmax) : 0.f;
    float den = e;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    if (lane < p.K) renorm[(int64_t)i * p.K + lane] = e / den;
  }
}

// Vocab tiles per block: the smallest makespan in tile units, counting one
// extra tile per block for pipeline fill and the unoverlapped last epilogue.
int pick_tiles_per_chunk(int n_mtiles, int n_vtiles, int n_sm) {
  int best = n_vtiles;
  long best_cost = -1;
  for (int tpc = 1; tpc <= n_vtiles; ++tpc) {
    const long chunks = (n_vtiles + tpc - 1) / tpc;
    const long blocks = chunks * n_mtiles;
    const long waves = (blocks + n_sm - 1) / n_sm;
    const long cost = waves * (tpc + 1);
    if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = tpc; }
  }
  return best;
}

}  // namespace

size_t score_workspace_size(int32_t M, int32_t d, int32_t V, int32_t K) {
  return score_layout(M, d, V, K).total;
}

mis_status_t launch_score(const ScoreArgs& a, void* stream) {
  const ScoreLayout L = score_layout(a.M, a.d, a.V, a.K);
  if (a.ws_bytes < L.total) return MIS_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  if (a.M == 0)   // no kernel runs: clear the status words here
    return cudaMemsetAsync(ws, 0, 8, st) == cudaSuccess ? MIS_OK : MIS_ERR_CUDA;

  __nv_bfloat16* gathered = reinterpret_cast<__nv_bfloat16*>(ws + L.gathered);
  int32_t* bad = reinterpret_cast<int32_t*>(ws + L.bad);
  if (launch_pdl(mis_gather_rows_kernel, dim3(L.m_pad), dim3(128), 0, st,
                 static_cast<const __nv_bfloat16*>(a.hidden), a.hidden_stride, a.T, a.delim, a.M,
                 a.d, gathered, bad, status) != cudaSuccess)
    return MIS_ERR_CUDA;

  bool ok = true;
  const uint64_t adims[2] = {(uint64_t)a.d, (uint64_t)L.m_pad};
  const uint64_t astr[1] = {(uint64_t)a.d * 2};
  const uint32_t abox[2] = {(uint32_t)kKStep, (uint32_t)kItemTile};
  const uint64_t wdims[2] = {(uint64_t)a.d, (uint64_t)a.V};
  const uint64_t wstr[1] = {(uint64_t)a.d * 2};
  const uint32_t wbox[2] = {(uint32_t)kKStep, (uint32_t)kVocabTile};
  CUtensorMap am = make_tmap_bf16(gathered, 2, adims, astr, abox, &ok);
  CUtensorMap wm = make_tmap_bf16(a.w_lm, 2, wdims, wstr, wbox, &ok);
  if (!ok) return MIS_ERR_CUDA;

  const int n_mtiles = L.m_pad / kItemTile;
  const int sms = num_sms();
  ScoreParams p;
  p.M = a.M; p.V = a.V; p.K = a.K;
  p.n_vtiles = L.n_vtiles;
  // one item tile and more vocabulary tiles than SMs: HBM-bound on W_lm; the
  // tiles go out from a counter so that every SM streams until the end.
  // Otherwise fixed runs of tiles, item tiles side by side in the grid so the
  // blocks sharing a W_lm tile run together and read it once through L2.
  p.dynamic = (n_mtiles == 1 && L.n_vtiles > sms) ? 1 : 0;
  p.ctr = status + 2;
  p.tiles_per_chunk = p.dynamic ? 0 : pick_tiles_per_chunk(n_mtiles, L.n_vtiles, sms);
  p.n_chunks = p.dynamic ? sms : (L.n_vtiles + p.tiles_per_chunk - 1) / p.tiles_per_chunk;
  p.n_parts = p.dynamic ? L.n_vtiles : p.n_chunks;
  p.n_kb = a.d / kKStep;
  p.w_lm = static_cast<const uint8_t*>(a.w_lm);
  // L2 prefetch of W_lm before the wait: only when the whole grid is one wave
  // (later waves start after the previous kernel anyway, where a prefetch
  // would only compete with the stream), about 32 MB in all, a quarter of L2
  {
    const int64_t blocks = (int64_t)n_mtiles * p.n_chunks;
    p.pf_bytes = 0;
    if (blocks <= sms) {
      const size_t per = ((size_t)32 << 20) / (size_t)p.n_chunks;
      p.pf_bytes = (uint32_t)std::min<size_t>(per & ~(size_t)65535, (size_t)1 << 30);
    }
  }
  for (int l = 0; l < 16; ++l) p.labels[l] = l < a.K ? a.labels[l] : -1;
  p.part = reinterpret_cast<float*>(ws + L.part);
  p.zlab = reinterpret_cast<float*>(ws + L.zlab);
  p.bad = bad;
  p.status = status;
  p.wait_ns = wait_limit_ns();
  p.stall = (inject_stall_mask() >> 1) & 1u;

  if (n_mtiles >= 2 && !p.dynamic) {
    // item tiles in pairs on SM pairs; each CTA loads half of a W_lm tile
    const uint32_t wbox2[2] = {(uint32_t)kKStep, (uint32_t)(kVocabTile / 2)};
    CUtensorMap wm2 = make_tmap_bf16(a.w_lm, 2, wdims, wstr, wbox2, &ok);
    if (!ok) return MIS_ERR_CUDA;
    if (!kernel_attr_once(reinterpret_cast<const void*>(mis_score_partial_pair_kernel), kPairSmem))
      return MIS_ERR_CUDA;
    if (launch_pdl(mis_score_partial_pair_kernel, dim3(n_mtiles, p.n_chunks), dim3(256),
                   kPairSmem, st, am, wm2, p) != cudaSuccess)
      return MIS_ERR_CUDA;
  } else {
    if (!kernel_attr_once(reinterpret_cast<const void*>(mis_score_partial_kernel), kSmem))
      return MIS_ERR_CUDA;
    if (launch_pdl(mis_score_partial_kernel, dim3(n_mtiles, p.n_chunks), dim3(256), kSmem, st,
                   am, wm, p) != cudaSuccess)
      return MIS_ERR_CUDA;
  }
  return launch_pdl(mis_score_combine_kernel, dim3((a.M + 3) / 4), dim3(128), 0, st, p,
                    a.out_logprobs, a.out_renorm) == cudaSuccess
             ? MIS_OK
             : MIS_ERR_CUDA;
}

}  // namespace mis

// ---------------------------------------------------------------------------
// Allocation-free label scoring (mis_label_scores_noalloc).
//
// Some callers of this library cannot call cudaMalloc: for example a plugin
// running inside an inference engine that has already reserved all free
// device memory for its own pools (KV cache, activations) and hands out no
// allocator, or a latency-critical path that must not pay the implicit
// device-wide synchronisation cudaMalloc/cudaFree can cause. They cannot
// provide the scoring workspace either, so this entry point keeps it in one
// file-scope device array of MIS_NOALLOC_SCRATCH_BYTES instead.
//
// Costs and rules of that choice:
//  * every GPU that loads this library holds the array until the process
//    exits;
//  * the device address is looked up once per device (cudaGetSymbolAddress,
//    with that device current) on the first call made on that device, so
//    make that first call before any stream capture;
//  * all calls on a device share the array and it keeps the last call's
//    contents: calls that overlap on the GPU (other streams, or host threads
//    without stream ordering between them) race and corrupt each other.
//    Each call clears the status words first and rewrites everything else it
//    reads (gathered rows including the zero padding, every (item, chunk)
//    pair, every label logit) before reading it.
// ---------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_noalloc_scratch[MIS_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (set up once).
mis_status_t noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MIS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MIS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MIS_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return MIS_OK;
}

}  // namespace

extern "C" mis_status_t mis_label_scores_noalloc(
    const void* hidden, int64_t hidden_row_stride, int32_t T, const void* w_lm, int32_t d,
    int32_t V, const int32_t* delim_positions, int32_t M, const int32_t* label_token_ids,
    int32_t K, float* out_logprobs, float* out_renorm, uint32_t* device_status, void* stream) {
  using namespace mis;
  // the same argument rules as mis_label_scores
  if (M < 0 || T < 1 || V < 1 || d < 1 || K < 1) return MIS_ERR_INVALID_ARG;
  if (K > 16) return MIS_ERR_UNSUPPORTED;
  if (d % 64 || d > 8192) return MIS_ERR_UNSUPPORTED;
  if (!label_token_ids) return MIS_ERR_INVALID_ARG;
  for (int l = 0; l < K; ++l)
    if (label_token_ids[l] < 0 || label_token_ids[l] >= V) return MIS_ERR_INVALID_ARG;
  auto misaligned = [](const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0;
  };
  if (M > 0) {
    if (!hidden || !w_lm || !delim_positions || !out_logprobs) return MIS_ERR_INVALID_ARG;
    if (misaligned(hidden, 16) || misaligned(w_lm, 16)) return MIS_ERR_INVALID_ARG;
    if (misaligned(delim_positions, 4) || misaligned(out_logprobs, 4) ||
        misaligned(out_renorm, 4) || misaligned(device_status, 4))
      return MIS_ERR_INVALID_ARG;
    if (hidden_row_stride < d || (hidden_row_stride & 7)) return MIS_ERR_SHAPE;
  }
  // sizes whose scratch would not fit the static array are refused
  if (score_workspace_size(M, d, V, K) > (size_t)MIS_NOALLOC_SCRATCH_BYTES)
    return MIS_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  mis_status_t st = noalloc_scratch(&scratch);
  if (st != MIS_OK) return st;
  ScoreArgs a;
  a.hidden = hidden; a.hidden_stride = hidden_row_stride; a.T = T;
  a.w_lm = w_lm; a.d = d; a.V = V;
  a.delim = delim_positions; a.M = M;
  for (int l = 0; l < 16; ++l) a.labels[l] = l < K ? label_token_ids[l] : -1;
  a.K = K;
  a.out_logprobs = out_logprobs; a.out_renorm = out_renorm;
  a.workspace = scratch; a.ws_bytes = MIS_NOALLOC_SCRATCH_BYTES;
  try {
    st = launch_score(a, stream);
  } catch (...) {
    return MIS_ERR_CUDA;
  }
  if (st == MIS_OK && device_status &&
      cudaMemcpyAsync(device_status, scratch, 2 * sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MIS_ERR_CUDA;
  return st;
}
