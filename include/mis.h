/*
 * mis.h — C ABI of the GB300 (sm_103a) Multiple-Item Scoring prefill hot path.
 *
 * Multiple-Item Scoring (MIS) packs one shared prefix and N candidate items
 * into one sequence and scores every item in a single prefill pass:
 *
 *     <prefix><DELIM><item 1><DELIM><item 2><DELIM> ... <item N><DELIM>
 *
 * ("Turbocharging LinkedIn's recommendation systems with SGLang", section
 * "Multi-item-scoring: Our innovation with SGLang"; "From Generation to
 * Scoring: Scaling LLM-Based Semantic Labeling at LinkedIn", Section 4.1,
 * eq. 3). Under the mask of eq. (4) of the latter, prefix tokens attend
 * causally to each other, every item token attends to the whole prefix and
 * causally inside its own item, never to another item. The label readout of
 * its Section 3.3 (eq. 2) takes the next-token distribution at each item's
 * readout row; "Scaling JEV-like Decision Models with SGLang" (section "Why a
 * Decision Workload Deserves a Scoring Interface") fixes that it is normalised
 * over the full vocabulary before the requested label columns are read.
 *
 * Conventions for every call
 *   - Every function returns mis_status_t; no exception or C++ type crosses
 *     the boundary. mis_status_string() names a code.
 *   - "device" pointers are CUDA global-memory addresses on the current
 *     device; "host" pointers are ordinary CPU memory. The caller owns every
 *     buffer, device or host, and allocates all of them; the library
 *     allocates no device memory. The only library-owned object is the
 *     host-side plan struct of mis_plan_create().
 *   - Calls that take a stream are stream-ordered and asynchronous: they
 *     enqueue work on `stream` (a cudaStream_t passed as void*, NULL = the
 *     legacy default stream) and return. Host input arrays may be reused as
 *     soon as the call returns. Device inputs are never modified.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and leave outputs untouched. Faults found on the device (an index out
 *     of range, a wait that ran out of time) are recorded in a status word at
 *     the start of the call's workspace; read it with mis_get_device_status().
 *   - Indices, lengths and counts are int32 (packed length T < 2^31).
 *   - bf16 tensors are IEEE bfloat16 stored as uint16.
 */
#ifndef MIS_GB300_H
#define MIS_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MIS_ABI_VERSION 2

typedef enum {
  MIS_OK = 0,
  MIS_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, bad count, bad id   */
  MIS_ERR_SHAPE = 2,          /* inconsistent lengths / offsets / strides      */
  MIS_ERR_UNSUPPORTED = 3,    /* valid but not built (head_dim, K, d ...)      */
  MIS_ERR_WORKSPACE = 4,      /* workspace missing, misaligned or too small    */
  MIS_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed             */
  MIS_ERR_DEVICE_TIMEOUT = 6, /* a kernel wait ran out of time and bailed out  */
  MIS_ERR_DEVICE_INDEX = 7    /* a device-side index was out of range          */
} mis_status_t;

const char* mis_status_string(int status);
int mis_abi_version(void);

/* ------------------------------------------------------------------------
 * Layout (host). Packs B requests into the delimiter layout above.
 *
 * Inputs (host):
 *   prefix_tokens[B] — P_b, prefix tokens of request b, excluding the DELIM
 *   n_items[B]       — N_b >= 0 items of request b
 *   item_lens[sum N] — L_i >= 0 tokens of each item excluding its DELIM,
 *                      request after request
 * Outputs (host, caller-allocated):
 *   cu_seqlens[B+1]  — request b occupies packed rows [cu[b], cu[b+1])
 *   prefix_len[B]    — S_b = P_b + 1: the shared set Q of eq. (4) is the
 *                      prefix plus its leading DELIM
 *   item_ptr[B+1]    — items of request b are [item_ptr[b], item_ptr[b+1])
 *   item_offsets[M]  — absolute first row of item i's set I_i (its tokens
 *                      followed by its trailing DELIM); the set ends where the
 *                      next item starts, or at the request end
 *   delim_positions[M] — absolute row of item i's trailing DELIM, the row
 *                      that reads prefix + item i (the readout row)
 *   position_ids     — may be NULL; else [position_cap] receives the reused
 *                      positions of Section 4.1: 0..S_b-1 on Q, S_b + d at
 *                      offset d of every item set (all items start at S_b)
 * Errors: MIS_ERR_INVALID_ARG (null array, negative length, B < 1),
 *         MIS_ERR_SHAPE (T or a position would overflow int32, or
 *         position_cap < T).
 * ------------------------------------------------------------------------ */
mis_status_t mis_layout_size(int32_t B, const int32_t* prefix_tokens, const int32_t* n_items,
                             const int32_t* item_lens, int64_t* T_out, int64_t* M_out);

mis_status_t mis_build_layout(int32_t B, const int32_t* prefix_tokens, const int32_t* n_items,
                              const int32_t* item_lens, int32_t* cu_seqlens, int32_t* prefix_len,
                              int32_t* item_ptr, int32_t* item_offsets, int32_t* delim_positions,
                              int32_t* position_ids, int64_t position_cap);

/* ------------------------------------------------------------------------
 * Setwise (multi-marker) layout: the anchor-based setwise prompt of "Scaling
 * JEV-like Decision Models with SGLang", section "Benchmark: Fused-Choice vs.
 * Setwise Scoring". Request b is ONE plain causal sequence: its
 * query_tokens[b] query tokens, the tokens of its n_cands[b] candidates
 * (cand_lens, request after request), then one marker per candidate; the
 * marker rows are the readout rows, in candidate order, and each sees every
 * candidate (no item isolation). Attention runs with a plain causal plan
 * (prefix_len[b] = request length, item_ptr = NULL) and scoring with
 * mis_label_scores at marker_positions.
 *   cu_seqlens       — host [B+1] out
 *   prefix_len       — host [B] out (= request length)
 *   marker_positions — host [M] out, M = sum of n_cands (may be NULL when M = 0)
 *   position_ids     — host [T] out (0..len-1 per request) or NULL
 * A request with no query token and no candidate is MIS_ERR_SHAPE.
 * ------------------------------------------------------------------------ */
mis_status_t mis_setwise_layout_size(int32_t B, const int32_t* query_tokens,
                                     const int32_t* n_cands, const int32_t* cand_lens,
                                     int64_t* T_out, int64_t* M_out);
mis_status_t mis_build_setwise_layout(int32_t B, const int32_t* query_tokens,
                                      const int32_t* n_cands, const int32_t* cand_lens,
                                      int32_t* cu_seqlens, int32_t* prefix_len,
                                      int32_t* marker_positions, int32_t* position_ids,
                                      int64_t position_cap);

/* ------------------------------------------------------------------------
 * Attention descriptor (all arrays host memory, read during planning only).
 *   B, T         — requests and packed rows; cu_seqlens[B] must equal T
 *   Hq, Hkv      — query / key-value heads; Hq % Hkv == 0; query head h
 *                  reads kv head h / (Hq / Hkv)
 *   D            — head dim, 64 or 128
 *   scale        — softmax scale; 0 selects 1/sqrt(D)
 *   cu_seqlens   — [B+1], 0 = cu[0] < cu[1] < ... (every request non-empty)
 *   prefix_len   — [B], 1 <= S_b <= request length: rows [cu[b], cu[b]+S_b)
 *                  form Q. S_b = request length with no items is plain
 *                  causal attention.
 *   item_ptr     — [B+1] CSR into item_offsets, or NULL when no request
 *                  has items
 *   item_offsets — absolute first row of each item set, strictly increasing
 *                  inside a request, the first equal to cu[b] + S_b; each
 *                  set is non-empty and the last ends at cu[b+1]
 * ------------------------------------------------------------------------ */
typedef struct {
  int32_t B, T, Hq, Hkv, D;
  float scale;
  const int32_t* cu_seqlens;
  const int32_t* prefix_len;
  const int32_t* item_ptr;
  const int32_t* item_offsets;
} mis_attn_desc;

typedef struct mis_plan_s* mis_plan_t;

typedef struct {
  int64_t n_qtiles;        /* (request, 128-row query tile) pairs              */
  int64_t n_tiles;         /* non-empty (query tile, 128-key tile) blocks      */
  int64_t n_full;          /* ... of which every entry is visible              */
  int64_t n_partial;       /* ... of which some entries are masked             */
  int64_t n_causal_tiles;  /* blocks a causal mask of the same cu_seqlens keeps */
  int64_t visible_pairs;   /* unmasked (row, key) pairs, per head              */
  int64_t workspace_bytes; /* device workspace the plan occupies               */
  int64_t schedule;        /* MIS_SCHEDULE_PAIR or MIS_SCHEDULE_SPLIT          */
  int64_t n_units;         /* work units of the attention kernel: query tiles  */
                           /* x (Hq / 2) for pairs, x Hq for split             */
} mis_plan_stats;

/* Bytes of device workspace mis_plan_create() needs for this descriptor (0
 * when the descriptor is invalid; mis_plan_create() then says why). */
size_t mis_plan_workspace_size(const mis_attn_desc* desc);

/* Validate the descriptor, build the mask-aware tile schedule on the host
 * (per query tile: the key tiles of the prefix plus the band of its own
 * items, each flagged full or partial; fully masked tiles are never listed —
 * "From Generation to Scoring" Section 4.2; "Turbocharging ...", section
 * "FlashInfer changes"), and upload
 * it into `workspace` (device, 256-byte aligned, >= mis_plan_workspace_size
 * bytes) on `stream`. The workspace must stay untouched while the plan is in
 * use. *out receives a host-side handle, freed by mis_plan_destroy().
 * workspace == NULL (with ws_bytes == 0) makes a host-only plan: no device
 * call is made, stats and the tile map can be read, and launching it returns
 * MIS_ERR_WORKSPACE.
 * Errors: MIS_ERR_INVALID_ARG / MIS_ERR_SHAPE / MIS_ERR_UNSUPPORTED on the
 * descriptor, MIS_ERR_WORKSPACE, MIS_ERR_CUDA on the upload. */
mis_status_t mis_plan_create(const mis_attn_desc* desc, void* workspace, size_t ws_bytes,
                             void* stream, mis_plan_t* out);
mis_status_t mis_plan_get_stats(mis_plan_t plan, mis_plan_stats* out);
/* Canonical tile map: int32 quadruples (request, q-tile, k-tile, 1 = full /
 * 2 = partial) for every non-empty 128x128 block, sorted by (request, q-tile,
 * k-tile). Writes min(cap, n) quadruples to host_out (may be NULL when cap is
 * 0); *n_out receives n. */
mis_status_t mis_plan_tile_map(mis_plan_t plan, int32_t* host_out, size_t cap, size_t* n_out);
/* The attention kernel's unit walk (for inspection and tests): the unit each
 * walk position hands out, -1 where a block has none. Position kk * G + c
 * belongs to block c in pass kk (odd passes reversed), G = min(units, SMs);
 * the plan's unit u is query tile u / g, head group u % g with g = Hq / 2
 * (pair schedule) or Hq (split). Every unit appears exactly once. Writes
 * min(cap, n) entries to host_out (may be NULL when cap is 0); *n_out
 * receives n and *blocks_out (may be NULL) receives G. */
mis_status_t mis_plan_unit_walk(mis_plan_t plan, int32_t* host_out, size_t cap, size_t* n_out,
                                int32_t* blocks_out);
/* The key tiles the attention kernel runs (for inspection and tests), query
 * tile by query tile in the plan's work-list order: quadruples (request,
 * first query row, first key row c0, flags) with flags bit 0 = the tile
 * needs the element mask (128 key rows from c0 each). Rows are absolute
 * (the new-row axis offset by the cache for cached plans).
 * Writes min(cap, n) quadruples to host_out (may be NULL when cap is 0);
 * *n_out receives n. */
mis_status_t mis_plan_exec_tiles(mis_plan_t plan, int32_t* host_out, size_t cap, size_t* n_out);
mis_status_t mis_plan_destroy(mis_plan_t plan);

/* Reusable planner for a stream of batches. mis_plan_create() uploads the
 * plan from pageable memory, which CUDA turns into a synchronisation with
 * the stream; a planner instead owns two pinned host staging buffers (grown
 * on demand) and an event per buffer, so mis_planner_plan() only waits for
 * the upload issued two calls earlier (long finished in a steady loop) and
 * the host can plan the next batch while the device still works. Same
 * validation, workspace rules and result as mis_plan_create(); the returned
 * plan is freed with mis_plan_destroy() and must not outlive its workspace.
 * A planner is not thread-safe; destroy waits for its uploads. */
typedef struct mis_planner_s* mis_planner_t;
mis_status_t mis_planner_create(mis_planner_t* out);
/* extra_host / extra_bytes: an optional side payload (e.g. the batch's
 * readout rows) copied in the same transfer to workspace +
 * mis_plan_workspace_size(desc); ws_bytes must cover it. NULL / 0 for none. */
mis_status_t mis_planner_plan(mis_planner_t planner, const mis_attn_desc* desc, void* workspace,
                              size_t ws_bytes, const void* extra_host, size_t extra_bytes,
                              void* stream, mis_plan_t* out);
mis_status_t mis_planner_destroy(mis_planner_t planner);

/* ------------------------------------------------------------------------
 * MIS attention forward ("From Generation to Scoring", eq. 4 and Section
 * 4.2; "Turbocharging ...", section "FlashInfer changes").
 *   q   — device bf16, row j of head h at q[j*q_row_stride + h*D + 0..D-1]
 *   k,v — device bf16, [T, Hkv, D] with their own row strides
 *   o   — device bf16 output, o[j*o_row_stride + h*D + ...]
 *   lse — device fp32 [Hq, T] natural-log softmax normaliser of the scaled
 *         scores (lse[h*T + j]), or NULL
 * Strides are in elements; each must be >= Hq*D (q, o) or Hkv*D (k, v) and a
 * multiple of 8; q, k, v, o must be 16-byte aligned. O rows of one call are
 * written exactly once; nothing else in o changes.
 * The plan form runs a plan from mis_plan_create(); the one-shot form plans,
 * launches and frees the host plan in one call (workspace as for
 * mis_plan_create()).
 * ------------------------------------------------------------------------ */
mis_status_t mis_attention_fwd_plan(mis_plan_t plan, const void* q, const void* k, const void* v,
                                    void* o, float* lse, int64_t q_row_stride,
                                    int64_t k_row_stride, int64_t v_row_stride,
                                    int64_t o_row_stride, void* stream);

mis_status_t mis_attention_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                               int64_t q_row_stride, int64_t k_row_stride, int64_t v_row_stride,
                               int64_t o_row_stride, const mis_attn_desc* desc, void* workspace,
                               size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Items over a cached prefix: the prefix K/V of each request was computed
 * earlier and kept in a cache buffer: the in-batch prefix cache of
 * "Scaling LLM-Based Ranking Systems with Prefill-Only Optimization"
 * (Components table), which reuses query-prefix KV within one forward
 * pass, and the knock-knock second request of "Turbocharging LinkedIn's
 * recommendation systems with SGLang", which appends the items to a prefix prefilled while
 * retrieval ran). The new sequence holds only item sets; each item row sees
 * its request's cached prefix (all of it: the prefix precedes every item
 * token) and its own item causally, as eq. (4) of "From Generation to
 * Scoring" gives for item rows. Single-item scoring with prefix caching is
 * the same call with one item per request, all requests pointing at one
 * cache range.
 *   B, T, Hq, Hkv, D, scale — as in mis_attn_desc (T = rows of the new sequence)
 *   cu_seqlens   — [B+1] new-sequence rows of each request (items only)
 *   item_ptr     — [B+1] CSR into item_offsets; every request has >= 1 item
 *   item_offsets — new-sequence first row of each item set (the first of a
 *                  request equals cu_seqlens[b]); each set ends where the next
 *                  starts or at cu_seqlens[b+1]
 *   cache_start  — [B] first cache row of request b's prefix (its |Q| rows:
 *                  prefix tokens and the leading DELIM)
 *   cache_len    — [B] S_b >= 1; cache_start[b] + S_b <= cache_T
 *   cache_T      — rows of the cache K/V buffers
 * Plans are made with mis_cached_plan_create (same workspace rules as
 * mis_plan_create) and run with mis_attention_fwd_cached; mis_plan_get_stats
 * and mis_plan_destroy apply. Key tiles of mis_plan_tile_map: indices below
 * ceil(S_b/128) are the cache tiles of the request, the rest the new
 * sequence's 128-row tiles counted from the request's first new row.
 * ------------------------------------------------------------------------ */
typedef struct {
  int32_t B, T, Hq, Hkv, D;
  float scale;
  const int32_t* cu_seqlens;
  const int32_t* item_ptr;
  const int32_t* item_offsets;
  const int32_t* cache_start;
  const int32_t* cache_len;
  int32_t cache_T;
} mis_cached_desc;

size_t mis_cached_plan_workspace_size(const mis_cached_desc* desc);
mis_status_t mis_cached_plan_create(const mis_cached_desc* desc, void* workspace, size_t ws_bytes,
                                    void* stream, mis_plan_t* out);

/* Attention of the new rows over [cached prefix ; own item]. q, k, v, o as
 * in mis_attention_fwd_plan for the T new rows; k_cache / v_cache device
 * bf16 [cache_T, Hkv, D] with row strides kc_row_stride / vc_row_stride (the
 * same rules). lse (optional) is [Hq, T] over the new rows. A plan of the
 * other kind returns MIS_ERR_INVALID_ARG (and mis_attention_fwd_plan refuses
 * cached plans the same way). */
mis_status_t mis_attention_fwd_cached(mis_plan_t plan, const void* q, const void* k,
                                      const void* v, const void* k_cache, const void* v_cache,
                                      void* o, float* lse, int64_t q_row_stride,
                                      int64_t k_row_stride, int64_t v_row_stride,
                                      int64_t kc_row_stride, int64_t vc_row_stride,
                                      int64_t o_row_stride, void* stream);

/* ------------------------------------------------------------------------
 * Rotary position embedding of Q and K at the reused position ids of "From
 * Generation to Scoring" Section 4.1 (query 0..S-1, offset d of every item
 * set -> S + d, as mis_build_layout emits them), so that every item is
 * rotated exactly as in its own single-item prompt ("Turbocharging ...",
 * section "SGLang changes": positional encoding adjusted so each item aligns
 * with its single-item position). The step before mis_attention_fwd*.
 * Rotate-half form: for i < D/2 the pair (x[i], x[i + D/2]) of a row at
 * position p turns by p * base^(-2i/D) (base > 1; 1e6 for the Qwen3 family).
 *   q, k          — device bf16 [T, Hq, D] and [T, Hkv, D], row strides in
 *                   elements (>= H*D, multiples of 8), 16-byte aligned
 *   q_out, k_out  — device bf16 outputs in the same shapes; q_out == q and
 *                   k_out == k (same strides) rotate in place; other overlaps
 *                   are not allowed. q and q_out both NULL rotate K only (for
 *                   mis_attention_fwd_plan_rope, which rotates Q on load;
 *                   Hq is then only checked, >= 1); one of them NULL alone
 *                   is MIS_ERR_INVALID_ARG
 *   position_ids  — device int32 [T]
 * fp32 arithmetic (angles from inverse frequencies computed in fp64 on the
 * host), bf16 results rounded to nearest even. One kernel launch, stream
 * ordered; T = 0 enqueues nothing.
 * ------------------------------------------------------------------------ */
mis_status_t mis_rope_qk(const void* q, const void* k, void* q_out, void* k_out,
                         int64_t q_row_stride, int64_t k_row_stride, int64_t q_out_row_stride,
                         int64_t k_out_row_stride, int32_t T, int32_t Hq, int32_t Hkv, int32_t D,
                         const int32_t* position_ids, double base, void* stream);

/* ------------------------------------------------------------------------
 * Rotary embedding of K alone at a plan's reused position ids (the same ids
 * mis_build_layout emits, derived on the device from the plan: rows of the
 * shared set at 0..S-1, row d of every item set at S + d), the companion of
 * mis_attention_fwd_plan_rope: no position ids travel to the device.
 * Rotate-half form and precision as mis_rope_qk.
 *   plan          — a plan with its device workspace (mis_plan_create or the
 *                   planner); packed or cached (K of the new rows)
 *   k, k_out      — device bf16 [T, Hkv, D], row strides in elements (>=
 *                   Hkv*D, multiples of 8), 16-byte aligned; k_out == k with
 *                   equal strides rotates in place
 * One kernel launch (one block per 128-row query tile), stream ordered after
 * the plan upload.
 * ------------------------------------------------------------------------ */
mis_status_t mis_rope_k_plan(mis_plan_t plan, const void* k, void* k_out, int64_t k_row_stride,
                             int64_t k_out_row_stride, double base, void* stream);

/* ------------------------------------------------------------------------
 * mis_attention_fwd_plan with the rotary embedding of Q fused in: Q arrives
 * unrotated and each unit's Q tile is turned in shared memory right after it
 * loads, at the row's reused position id ("From Generation to Scoring"
 * Section 4.1: rows of the shared set at 0..S-1, row d of every item set at
 * S + d; exactly the ids mis_build_layout emits), derived from the plan, so
 * every item is rotated as in its own single-item prompt ("Turbocharging
 * ...", section "SGLang changes"). Same rotate-half form as mis_rope_qk:
 * the pair (x[i], x[i + D/2]) turns by p * rope_base^(-2i/D), the angle in
 * fp32 (frequencies computed in fp64 on the host), its sine and cosine
 * evaluated on the device after an exact reduction to [-pi, pi]; the turned
 * tile is rounded to bf16 (nearest even) before the products, as a rotated
 * Q in memory would be. K must arrive rotated already (mis_rope_k_plan on
 * the same plan, or mis_rope_qk with q = q_out = NULL and the layout's
 * position ids); V is not rotated.
 *   rope_base — > 1 (1e6 for the Qwen3 family)
 * Requests longer than 2^17 rows return MIS_ERR_UNSUPPORTED. Everything
 * else as mis_attention_fwd_plan (packed plans only; a cached plan returns
 * MIS_ERR_INVALID_ARG). Q in global memory is read, never written.
 * ------------------------------------------------------------------------ */
mis_status_t mis_attention_fwd_plan_rope(mis_plan_t plan, const void* q, const void* k,
                                         const void* v, void* o, float* lse,
                                         int64_t q_row_stride, int64_t k_row_stride,
                                         int64_t v_row_stride, int64_t o_row_stride,
                                         double rope_base, void* stream);

/* ------------------------------------------------------------------------
 * Label scoring at the readout rows ("From Generation to Scoring", Section
 * 3.3 and eq. 2; "Turbocharging ...", section "SGLang changes": an N x K
 * matrix of label log-probs; "Scaling JEV-like Decision Models with SGLang",
 * "Send a Scoring Request": apply_softmax normalises across labels per item).
 *   hidden          — device bf16 [T, d], row stride hidden_row_stride (>= d,
 *                     multiple of 8); the final-normed hidden states
 *   w_lm            — device bf16 [V, d] row-major LM head (row v = token v)
 *   delim_positions — device int32 [M], readout row of each item, in [0, T)
 *   label_token_ids — host int32 [K], 0 <= id < V, caller order, repeats ok
 *   out_logprobs    — device fp32 [M, K]: z_i[label] - logsumexp_v z_i[v],
 *                     z_i = W_lm h_i over the full vocabulary
 *   out_renorm      — device fp32 [M, K] softmax over the K label logits of
 *                     each item (eq. 2 when K = 2), or NULL
 * Constraints: d a multiple of 64 (<= 8192), 1 <= K <= 16, 1 <= V, M >= 0.
 * The full logits never reach global memory: each 128 x 256 logit tile lives
 * in tensor memory and leaves only a (max, sum-of-exp) pair per item.
 * Workspace: device, 256-byte aligned, >= mis_label_scores_workspace_size().
 * A readout row outside [0, T) sets MIS_ERR_DEVICE_INDEX in the workspace
 * status and scores a zero hidden row instead.
 * W_lm is treated as a weight: the LM-head kernel starts reading it (into
 * shared memory and L2) while the work enqueued on the stream before this
 * call is still finishing, so that work must not write W_lm (write it in
 * an earlier, completed step, or synchronise before the call). `hidden` and
 * `delim_positions` are read only after all earlier stream work completed.
 * ------------------------------------------------------------------------ */
size_t mis_label_scores_workspace_size(int32_t M, int32_t d, int32_t V, int32_t K);

mis_status_t mis_label_scores(const void* hidden, int64_t hidden_row_stride, int32_t T,
                              const void* w_lm, int32_t d, int32_t V,
                              const int32_t* delim_positions, int32_t M,
                              const int32_t* label_token_ids, int32_t K, float* out_logprobs,
                              float* out_renorm, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Device status of the last call that used `workspace` (a plan workspace or
 * a scoring workspace). Synchronises `stream`, then returns MIS_OK,
 * MIS_ERR_DEVICE_TIMEOUT or MIS_ERR_DEVICE_INDEX. Each call clears the word
 * when it starts.
 * ------------------------------------------------------------------------ */
mis_status_t mis_get_device_status(const void* workspace, void* stream);

/* Upper bound, in nanoseconds, on any single wait inside the kernels
 * (default 200 ms). A wait that runs out sets MIS_ERR_DEVICE_TIMEOUT, lets
 * every role of the block drain its own copies and tensor-memory work, frees
 * tensor memory and returns. Small values exist for tests of that path.
 * Process-wide; returns the previous value. */
uint64_t mis_set_wait_limit_ns(uint64_t ns);

/* Failure injection for tests, without a GPU fault. While bit 0 (attention)
 * or bit 1 (scoring) of `mask` is set, the tensor-core thread of every block
 * launched by those calls first waits on a barrier that nothing arrives on,
 * so the bounded wait runs out and the timeout path above runs for real:
 * MIS_ERR_DEVICE_TIMEOUT in the workspace status, outputs not written, the
 * context left usable. 0 (the default) turns it off. Process-wide; returns
 * the previous mask. */
uint32_t mis_inject_stall(uint32_t mask);

/* Attention schedule of plans created after the call (process-wide; returns
 * the previous mode, or -1 for an unknown mode, which changes nothing).
 *   MIS_SCHEDULE_AUTO  — the planner picks (default);
 *   MIS_SCHEDULE_PAIR  — a unit is one query tile for two query heads that
 *                        share a kv head; each of the block's two softmax
 *                        streams computes one head over every key tile;
 *   MIS_SCHEDULE_SPLIT — a unit is one query tile for one head; the streams
 *                        take alternate key tiles and merge their partial
 *                        (max, sum, O) in the epilogue: twice the units at
 *                        half the length, which fills the last wave of SMs
 *                        better, at twice the K/V tile loads per FLOP.
 * AUTO compares the two by the largest per-SM sum of unit costs under the
 * kernel's static unit order. PAIR needs an even Hq / Hkv; odd groups always
 * run SPLIT. The result is the same up to float rounding either way. */
#define MIS_SCHEDULE_AUTO 0
#define MIS_SCHEDULE_PAIR 1
#define MIS_SCHEDULE_SPLIT 2
int32_t mis_set_schedule(int32_t mode);

/* ------------------------------------------------------------------------
 * Allocation-free label scoring. The pages have no counterpart of this call;
 * it exists for callers that cannot call cudaMalloc, such as a plugin inside
 * an inference engine that has already reserved all free device memory and
 * offers no allocator, or a latency-critical path that must not take the
 * device-wide synchronisation cudaMalloc/cudaFree can cause.
 *
 * Same inputs, outputs and results as mis_label_scores(), but no workspace:
 * the scratch (gathered readout rows, per-chunk logsumexp pairs, label
 * logits, status words) lives in one static device array of
 * MIS_NOALLOC_SCRATCH_BYTES inside the library. The call allocates nothing
 * and calls no allocating routine.
 *   - Size limit: any (M, d, V, K) whose mis_label_scores_workspace_size() is
 *     at most MIS_NOALLOC_SCRATCH_BYTES (for example M <= 512 items with
 *     d <= 4096, V <= 262144, K <= 16); larger calls return
 *     MIS_ERR_UNSUPPORTED before anything is enqueued.
 *   - Every GPU that loads the library holds the array until process exit.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents. Calls that overlap on the GPU (different streams, or host
 *     threads without ordering) race and corrupt each other's results;
 *     serialise them on one stream.
 *   - device_status: optional device uint32[2] that receives this call's
 *     device status words after the kernels ([0] bit 1 = a wait timed out,
 *     bit 2 = a readout row was outside [0, T); [1] = first failing site);
 *     NULL skips the copy. There is no workspace to hand to
 *     mis_get_device_status(), so with NULL a readout row outside [0, T)
 *     (scored as a zero hidden row) and a timed-out wait go unreported:
 *     pass a status buffer wherever such errors must be seen.
 * ------------------------------------------------------------------------ */
#define MIS_NOALLOC_SCRATCH_BYTES (8650752) /* 8.25 MiB */

mis_status_t mis_label_scores_noalloc(const void* hidden, int64_t hidden_row_stride, int32_t T,
                                      const void* w_lm, int32_t d, int32_t V,
                                      const int32_t* delim_positions, int32_t M,
                                      const int32_t* label_token_ids, int32_t K,
                                      float* out_logprobs, float* out_renorm,
                                      uint32_t* device_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MIS_GB300_H */
