/*
 * ssa.h -- C ABI of the GB300 (sm_103a) sparse-attention decode library.
 *
 * One decode step of one sparse-attention layer, for a batch of requests:
 *
 *   ssa_index_topk          int8 indexer over a compressed per-page key slab,
 *                           then a fixed-shape top-k page selection
 *   ssa_ensure_resident     device-side LRU: bind every selected logical page
 *                           to a physical GPU slot, fetch misses from the
 *                           pinned host mirror over UVA (NVLink-C2C)
 *   ssa_remap_block_table   selected logical pages -> physical slots
 *   ssa_sparse_paged_decode GQA decode attention over the selected pages only
 *
 * and the write path that fills the cache:
 *
 *   ssa_store_kv_mirror     quantise (fp8) or pass through (bf16) new K/V,
 *                           write the pinned host mirror and, when resident,
 *                           the GPU slot; update the indexer slab
 *
 * Sources (web pages, cited by title and section):
 *   FreeToken PR #499 "host-RAM KV tier for sparse-attention models
 *     (--kv-host-pages)": "What", "Why this works for sparse attention",
 *     "Design", "Known limitations".
 *   FreeToken PR #525 "host-resident prefix tier for hybrid GDN models",
 *     conversation summary: mirror_store_quant, scale banks, select width.
 *   vLLM issue #33980 "[RFC]: Sparse attention KV cache offloading",
 *     "Motivation" and "Proposed Change".
 *
 * ---------------------------------------------------------------------------
 * Conventions for every call
 *   * Ownership: the caller allocates and owns every buffer.  Device buffers
 *     are plain device pointers; the host mirror is pinned host memory that
 *     the GPU can address (cudaHostAlloc / pinned torch tensors; on a
 *     unified-addressing system the host pointer is also the device pointer).
 *     The library allocates nothing and keeps no pointer after a call returns.
 *   * Streams: every call only enqueues work on `stream` (a cudaStream_t) and
 *     never synchronises the host, so a sequence of calls can be captured in
 *     a CUDA graph.  Calls on one stream are ordered; the caller orders
 *     streams.
 *   * Layers: every call takes a layer range [layer0, layer0 + n_layers).
 *     Cache arrays (ssa_cache) are indexed by absolute layer; per-call arrays
 *     (q, sel, phys, out, ...) hold n_layers consecutive layer slices, slice 0
 *     being layer0.  One launch covers the whole range.
 *   * Return value: SSA_OK, or a negative SSA_ERR_* found on the host before
 *     anything was enqueued (SSA_ERR_CUDA: a launch failed; the cudaError_t
 *     is kept for ssa_last_cuda_error()).
 *   * Device-detected problems set bits (atomicOr) in the caller's int32
 *     status word `status` (device memory, may be NULL): SSA_ST_*.  The word
 *     is never cleared by the library; the caller reads it when it chooses.
 *   * No kernel traps, asserts or waits without a bound: a wait that runs out
 *     sets SSA_ST_TIMEOUT and the kernel returns.
 * ---------------------------------------------------------------------------
 */
#ifndef SSA_H
#define SSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-compatible with cudaStream_t. */
typedef struct CUstream_st *ssa_stream_t;

enum {
  SSA_OK = 0,
  SSA_ERR_INVALID_ARG = -1,   /* null pointer, bad range, bad layout field   */
  SSA_ERR_POOL_TOO_SMALL = -2,/* pool_slots < min(batch*max_sel, logical)    */
  SSA_ERR_UNSUPPORTED = -3,   /* dtype, page size, head_dim, GQA group       */
  SSA_ERR_NO_MIRROR = -4,     /* a host tier call without mirror pointers    */
  SSA_ERR_CUDA = -5,          /* a CUDA launch or attribute query failed     */
  SSA_ERR_SCRATCH_LIMIT = -6  /* ssa_index_topk_static_scratch: the call needs
                                 more than SSA_STATIC_SCORE_ENTRIES scores     */
};

enum {
  SSA_ST_DROP = 1,            /* a selection did not fit max_sel (counted)   */
  SSA_ST_BAD_ID = 2,          /* logical page id or page index out of range  */
  SSA_ST_MISS_NO_MIRROR = 4,  /* a miss had no host mirror to fetch from     */
  SSA_ST_UNRESOLVED = 8,      /* a selected page had no slot at remap/decode */
  SSA_ST_BAD_POS = 16,        /* store positions not strictly increasing     */
  SSA_ST_TIMEOUT = 32,        /* a bounded device wait gave up               */
  SSA_ST_INTERNAL = 64        /* a kernel's own consistency check failed (its
                                 work was abandoned; report it as a bug)       */
};

enum { SSA_KV_BF16 = 0, SSA_KV_FP8_E4M3 = 1 };

/*
 * Shapes.  Validated by every call.
 *   page_size   P, tokens per page: 16, 32, 64 or 128
 *   n_q_heads   Hq;  n_kv_heads Hkv;  G = Hq / Hkv must be an integer, 1..8
 *   head_dim    D, must be 128
 *   kv_dtype    SSA_KV_BF16 or SSA_KV_FP8_E4M3
 *   n_layers    layers held by the cache arrays
 *   logical_pages  Lp, logical page ids per layer (0 .. Lp-1)
 *   pool_slots  S, physical GPU slots per layer
 *   batch       B requests;  max_pages n_max = block-table width
 *   block_topk  k >= 1;  max_sel W must equal 2*k + 8 (FreeToken PR #499,
 *               "Design": max_sel_pages sized from 2*block_topk + 8)
 */
typedef struct ssa_layout {
  int page_size, n_q_heads, n_kv_heads, head_dim;
  int kv_dtype;
  int n_layers, logical_pages, pool_slots;
  int batch, max_pages, block_topk, max_sel;
} ssa_layout;

/*
 * The paged KV cache and its residency state (all per layer, layer-major).
 *
 *   k_pool   [Lyr][S][Hkv][P][D]   bf16 values, or e4m3 codes
 *   v_pool   bf16: [Lyr][S][Hkv][P][D];  fp8: [Lyr][S][Hkv][D][P] (each KV
 *            head's page stored d-major, tokens contiguous, so the attention
 *            kernel reads 8-bit V with tokens along the reduction)
 *   k_scale, v_scale   [Lyr][S][P] fp32 per-token scales (fp8 only; else NULL)
 *   k_mirror, v_mirror, k_scale_mirror, v_scale_mirror: the same per-page
 *            blocks indexed by logical page, [Lyr][Lp][...], in pinned host
 *            memory; all four NULL means no host tier.  Mirror bytes equal
 *            pool bytes for every bound slot (FreeToken PR #525: the mirror
 *            holds the codes and scales after quantisation).
 *   slab       [Lyr][Lp][Hkv][D] int8 page-mean key codes (the indexer slab)
 *   slab_scale [Lyr][Lp] fp32, the per-page symmetric scale amax/127
 *   slab_sum   [Lyr][Lp][Hkv][D] fp32 running key sums (token order)
 *   slab_cnt   [Lyr][Lp] int32 tokens summed
 *   slot_of  [Lyr][Lp]  physical slot of a logical page, or -1
 *   page_of  [Lyr][S]   logical page held by a slot, or -1 (free)
 *   last_use [Lyr][S]   clock value of the slot's last use, -1 never
 *   clock    [Lyr]      ensure steps taken
 * Device pointers except the mirrors.  All 256-byte aligned, except that
 * scale arrays need 16 bytes.
 */
typedef struct ssa_cache {
  void *k_pool, *v_pool;
  float *k_scale, *v_scale;
  void *k_mirror, *v_mirror;
  float *k_scale_mirror, *v_scale_mirror;
  int8_t *slab;
  float *slab_scale;
  float *slab_sum;
  int32_t *slab_cnt;
  int32_t *slot_of, *page_of, *last_use, *clock;
} ssa_cache;

/* Bytes of scratch (device memory, 256-byte aligned) that ssa_index_topk,
 * ssa_ensure_resident and ssa_sparse_paged_decode need for any layer range
 * of this layout.  The calls use disjoint parts of it.  Zero the workspace
 * once before its first use: ssa_sparse_paged_decode keeps per-unit split
 * counters in it, and every call that completes leaves them zero again (a
 * call that reported SSA_ST_TIMEOUT may not: zero the workspace again).
 * 0 on a bad layout. */
size_t ssa_workspace_size(const ssa_layout *lay);

/*
 * Reset the residency state of every layer (FreeToken PR #499, "What": the
 * GPU's slots cache logical pages, least recently used out first).
 *   identity = 0: empty pool (slot_of = page_of = last_use = -1, clock 0);
 *   identity = 1: fully resident, slot s holds logical page s for
 *                 s < min(S, Lp), last_use -1, clock 0.
 * Also zeroes slab, slab_scale, slab_sum and slab_cnt.
 */
int ssa_lru_init(const ssa_layout *lay, const ssa_cache *c, int identity,
                 ssa_stream_t stream);

/*
 * a0 -- store K/V through the write-through mirror (FreeToken PR #499,
 * "Design": each stored token also goes to pinned host memory, so evicting a
 * slot never needs a write-back; FreeToken PR #525: with fp8 the host copy
 * holds the quantised codes and their scales, byte for byte the pool's).
 *   k, v   [n_layers][T][Hkv][D] bf16, device
 *   pos    [T] int64 logical token ids, page = pos / P, row j = pos % P;
 *          strictly increasing within the call (SSA_ST_BAD_POS otherwise),
 *          each position stored once over the cache's lifetime
 * A call holds any run of tokens: a prefill chunk, or the one token per
 * request a decode step appends; a page may be filled over many calls, and
 * its slab row then equals that of one call storing the same tokens.
 * fp8: per token and tensor, s = max|x| / 448 over all KV heads (1 if the
 * token is all zero), code = e4m3(x / s) rounded to nearest even,
 * saturating.  Writes the mirror always (when present) and the pool slot
 * when the page is resident.  Slab: adds each token's bf16 keys to slab_sum
 * in token order, counts them, and re-quantises the touched pages:
 * mean = sum / count, s = max|mean| / 127, code = clamp(rint(mean/s), +-127)
 * (all zero when max|mean| = 0).  Out-of-range pages: SSA_ST_BAD_ID.
 */
int ssa_store_kv_mirror(const ssa_layout *lay, const ssa_cache *c, int layer0, int n_layers,
                        const void *k, const void *v, const int64_t *pos, int T,
                        int32_t *status, ssa_stream_t stream);

/*
 * a1 + a2 -- indexer and top-k page selection (FreeToken PR #499, "Why this
 * works for sparse attention": every attend step first runs top-k block
 * selection over the compressed, GPU-resident slab, fixed shape; "Design":
 * compact_selected_pages with a drop counter).
 *   q           [n_layers][B][Hq][D] bf16, device
 *   block_table [B][n_max] int32 logical page ids of each request's pages
 *   seq_lens    [B] int32 tokens per request; n_b = ceil(seq_len / P) pages
 *   sel         [n_layers][B][W] int32 out: selected page indices (into the
 *               request's block-table row), ascending, -1 padded
 *   n_sel       [n_layers][B] int32 out
 *   scores_opt  [n_layers][B][n_max] int32 out or NULL; INT32_MIN past n_b
 * q is quantised per request: s = max|q| / 127 over all Hq*D values,
 * q8 = clamp(rint(q/s), +-127).  Score of page p (exact int32):
 *   S[p] = sum_hq sum_d q8[hq][d] * slab[bt[p]][hq / G][d].
 * Selection: the k best of pages [0, n_b - 1) by (score desc, page asc),
 * plus page n_b - 1 always; all pages when n_b - 1 <= k.  Selections that
 * would not fit W are dropped and flagged SSA_ST_DROP (cannot happen when
 * W = 2k + 8).  One launch: the last CTA to finish scoring a (layer,
 * request) row selects over it.  ws: ssa_workspace_size bytes, zeroed once
 * (required; it holds the per-row tickets).
 */
int ssa_index_topk(const ssa_layout *lay, const ssa_cache *c, int layer0, int n_layers,
                   const void *q, const int32_t *block_table, const int32_t *seq_lens,
                   int32_t *sel, int32_t *n_sel, int32_t *scores_opt, int32_t *status,
                   void *ws, ssa_stream_t stream);

/*
 * a3 + a4 -- LRU ensure and miss fetch (FreeToken PR #499, "Design": the
 * LRU runs on the device with fixed shapes, so it can sit in a CUDA graph;
 * evicting only rebinds a slot; misses are copied host -> device; FreeToken
 * PR #525: the copy includes the fp8 scales, and the pool is sized so that
 * the whole batch's selection fits).
 * Per layer, in this order:
 *   1. U = distinct logical ids bt[b][sel[b][i]] of the batch, ascending;
 *   2. hits are touched: last_use[slot] = clock;
 *   3. misses (ascending id) take victims in order: free slots by ascending
 *      slot id, then bound slots not touched this step by ascending
 *      (last_use, slot); the victim's old page loses its slot;
 *   4. each miss's K, V (and fp8 scales) are copied mirror -> slot;
 *   5. clock += 1.
 *   sel                    [n_layers][B][W] from ssa_index_topk
 *   miss_page_opt, miss_slot_opt  [n_layers][B*W] int32 out or NULL
 *   n_miss_opt             [n_layers] int32 out or NULL
 * Requires pool_slots >= min(B*W, Lp) (SSA_ERR_POOL_TOO_SMALL).  A miss
 * without a mirror is bound but not fetched: SSA_ST_MISS_NO_MIRROR.
 */
int ssa_ensure_resident(const ssa_layout *lay, const ssa_cache *c, int layer0, int n_layers,
                        const int32_t *sel, const int32_t *block_table,
                        int32_t *miss_page_opt, int32_t *miss_slot_opt, int32_t *n_miss_opt,
                        int32_t *status, void *ws, ssa_stream_t stream);

/*
 * a3 + a4 + a5 in one call: ssa_ensure_resident, whose LRU kernel also
 * writes the remapped table once every selected page has its slot -- the
 * same phys as ssa_remap_block_table (FreeToken PR #499, "Design": after
 * ensure the block table is translated logical -> physical), one launch
 * fewer per step.
 *   phys [n_layers][B][W] int32 out (required)
 */
int ssa_ensure_remap(const ssa_layout *lay, const ssa_cache *c, int layer0, int n_layers,
                     const int32_t *sel, const int32_t *block_table, int32_t *phys,
                     int32_t *miss_page_opt, int32_t *miss_slot_opt, int32_t *n_miss_opt,
                     int32_t *status, void *ws, ssa_stream_t stream);

/*
 * ssa_ensure_remap in two calls, so that the host-link copy of one layer
 * range can run while the attention of another range reads its pages
 * (vLLM RFC #33980, "Motivation": the load time is what has to be hidden;
 * FreeToken PR #499, "Design": ensure, then copy, then attend, per layer).
 *   ssa_ensure_remap_bind: steps 1-3 and 5 of ssa_ensure_resident and the
 *     remap of ssa_ensure_remap -- the residency state, phys and the miss
 *     lists are final -- but nothing is copied;
 *   ssa_fetch_misses: step 4 for the layers [layer0, layer0 + n_layers):
 *     each listed miss's K, V (and fp8 scales) mirror -> slot.  Any split of
 *     a bind call's range into fetch calls (lists offset to the first layer
 *     of each) gives the bytes of the one ssa_ensure_remap call.
 * Between the two, a missed page's slot holds stale bytes while phys already
 * names it: the attention over a layer goes after that layer's fetch (same
 * stream, or an event), and no other call on those layers goes between.
 *   phys           [n_layers][B][W] int32 out (bind)
 *   miss_page, miss_slot  [n_layers][B*W] int32, out (bind) / in (fetch)
 *   n_miss         [n_layers] int32, out (bind) / in (fetch)
 * The lists are required (no workspace default).  The fetch needs the host
 * mirror (SSA_ERR_NO_MIRROR); the bind flags a miss without one on the
 * device, as ssa_ensure_resident does.
 */
int ssa_ensure_remap_bind(const ssa_layout *lay, const ssa_cache *c, int layer0, int n_layers,
                          const int32_t *sel, const int32_t *block_table, int32_t *phys,
                          int32_t *miss_page, int32_t *miss_slot, int32_t *n_miss,
                          int32_t *status, ssa_stream_t stream);
int ssa_fetch_misses(const ssa_layout *lay, const ssa_cache *c, int layer0, int n_layers,
                     const int32_t *miss_page, const int32_t *miss_slot, const int32_t *n_miss,
                     int32_t *status, ssa_stream_t stream);

/*
 * The miss fetch folded into the attention: ssa_ensure_remap_deferred runs
 * the ensure's state update and remap (a3, a5) but copies nothing; its phys
 * marks each page this call bound (a miss) as -2 - slot.  Then
 * ssa_sparse_paged_decode_fetch runs the attention on that phys: a marked
 * page is read from the pinned host mirror inside the attention kernel (the
 * host-tail path), used, and written into its slot as it streams past, so
 * the host-link reads overlap the attention over the resident pages instead
 * of preceding it (FreeToken PR #499, "Design": ensure, then copy, then
 * attend; vLLM RFC #33980, "Motivation": the load time is what has to be
 * hidden).  The residency state, the miss lists, the pool bytes afterwards
 * and the outputs are those of ssa_ensure_remap + ssa_sparse_paged_decode.
 * Between the two calls the marked slots hold stale bytes: nothing else may
 * read them, and the pair must not be split across other calls on the
 * cache.  Both require the host mirror (SSA_ERR_NO_MIRROR).
 *   phys [n_layers][B][W] int32 out / in: slot, -2 - slot (marked), or -1
 *   block_table (fetch): as for ssa_index_topk, for the marked pages' ids
 */
int ssa_ensure_remap_deferred(const ssa_layout *lay, const ssa_cache *c, int layer0,
                              int n_layers, const int32_t *sel, const int32_t *block_table,
                              int32_t *phys, int32_t *miss_page_opt, int32_t *miss_slot_opt,
                              int32_t *n_miss_opt, int32_t *status, void *ws,
                              ssa_stream_t stream);
int ssa_sparse_paged_decode_fetch(const ssa_layout *lay, const ssa_cache *c, int layer0,
                                  int n_layers, const void *q, const int32_t *sel,
                                  const int32_t *phys, const int32_t *block_table,
                                  const int32_t *seq_lens, float sm_scale, void *out,
                                  int32_t *status, void *ws, ssa_stream_t stream);

/*
 * Residency shared by the layers of a call (FreeToken PR #499, "Design": one
 * launch copies a page's K and V for all the sparse-attention layers).  The
 * layers [layer0, layer0 + n_layers) share ONE LRU state, layer0's slot_of /
 * page_of / last_use / clock (the other layers' state arrays are not used):
 *   1. U = distinct logical ids selected by any layer of the range, ascending;
 *   2-5. as ssa_ensure_resident, on that one state: hits touched, misses take
 *      free slots then untouched slots by (last_use, slot), rebind, clock + 1;
 *      each miss's K, V (and fp8 scales) are copied into the same slot of
 *      EVERY layer's pool (one launch for all layers);
 *   then phys [n_layers][B][W] = slot_of[layer0][bt[b][sel]] for every layer.
 *   miss_page_opt, miss_slot_opt [n_layers * B * W] int32 out or NULL
 *   n_miss_opt  [1] int32 out or NULL: misses of the call
 * Requires n_layers * B * W <= 16384 (SSA_ERR_UNSUPPORTED) and pool_slots >=
 * min(n_layers * B * W, logical_pages) (SSA_ERR_POOL_TOO_SMALL).  Use one
 * residency mode per cache: this call and ssa_ensure_resident / ssa_ensure_remap
 * keep different state.
 */
int ssa_ensure_remap_shared(const ssa_layout *lay, const ssa_cache *c, int layer0,
                            int n_layers, const int32_t *sel, const int32_t *block_table,
                            int32_t *phys, int32_t *miss_page_opt, int32_t *miss_slot_opt,
                            int32_t *n_miss_opt, int32_t *status, void *ws,
                            ssa_stream_t stream);

/*
 * Top-k preload (vLLM RFC #33980, "Motivation" point 2 and "Proposed Change":
 * "Topk KV preload" -- adjacent decode steps select largely the same pages,
 * so a former top-k can drive a fetch that overlaps the current step's
 * compute, leaving only the residual misses to load once the actual top-k
 * is known).  Run after a step's ssa_ensure_resident, on that step's scores:
 *   1. candidates, per request: the top (width - 1) pages of [0, n_b - 1) by
 *      (score desc, page asc) plus page n_b - 1 (all pages when
 *      n_b - 1 <= width - 1) -- the selection rule with k = width - 1;
 *   2. per layer, U = the distinct logical ids of the batch's candidates;
 *      with e = clock - 1 (the epoch of the step's ensure):
 *   3. resident ids of U are touched: last_use = e;
 *   4. the other ids of U, ascending, take victims in order: free slots by
 *      ascending slot id, then bound slots with last_use < e by ascending
 *      (last_use, slot) -- so the pages the step's attention reads are never
 *      evicted; ids left over when no victim remains are not fetched;
 *   5. each bound id gets last_use = e and its K, V (and fp8 scales) are
 *      copied mirror -> slot; the clock is not advanced.
 * The next ssa_ensure_resident then finds the fetched pages resident.
 *   scores        [n_layers][B][n_max] int32: the step's scores_opt from
 *                 ssa_index_topk; must not change until this call completes
 *   width         candidates per request, 1 <= width <= max_sel
 *   fetch_page_opt, fetch_slot_opt  [n_layers][B*W] int32 out or NULL
 *   n_fetch_opt   [n_layers] int32 out or NULL: pages fetched per layer
 * ws is required (the candidates and fetch lists live in a part of it that
 * no other call uses).  Ordering: after the step's ssa_remap_block_table
 * (which reads the state this call changes) and before the next step's
 * ssa_ensure_resident; it may run on a second stream concurrently with the
 * step's ssa_sparse_paged_decode (the slots it reads are never victims) and
 * the next step's ssa_index_topk (which must write its scores elsewhere).
 * SSA_ERR_POOL_TOO_SMALL as ssa_ensure_resident.
 */
int ssa_prefetch_pages(const ssa_layout *lay, const ssa_cache *c, int layer0, int n_layers,
                       const int32_t *scores, const int32_t *block_table,
                       const int32_t *seq_lens, int width, int32_t *fetch_page_opt,
                       int32_t *fetch_slot_opt, int32_t *n_fetch_opt, int32_t *status, void *ws,
                       ssa_stream_t stream);

/*
 * a5 -- block-table translation (FreeToken PR #499, "Design": after ensure
 * the block table is translated logical -> physical and attention runs on
 * it unmodified).
 *   phys [n_layers][B][W] int32 out: slot_of[bt[b][sel]] or -1 for padding;
 *   a selected page without a slot gives -1 and SSA_ST_UNRESOLVED.
 */
int ssa_remap_block_table(const ssa_layout *lay, const ssa_cache *c, int layer0, int n_layers,
                          const int32_t *sel, const int32_t *block_table, int32_t *phys,
                          int32_t *status, ssa_stream_t stream);

/*
 * a6 + a7 -- paged GQA decode attention over the selected pages only
 * (FreeToken PR #499, "Design": qsa_sparse_paged_attention runs on the
 * remapped table).  For request b and query head hq (KV head h = hq / G):
 *   out[b][hq] = sum_t softmax_t(sm_scale * q[b][hq] . K[t]) V[t]
 * over tokens t = p*P + j of the pages p = sel[b][i] with phys[b][i] >= 0
 * and t < seq_lens[b]; K[t] = code * k_scale[t] for fp8 (V likewise).
 * Entries with sel < 0 are padding; sel >= 0 with phys < 0 are skipped and
 * flagged SSA_ST_UNRESOLVED.  A request with no token gets zeros.
 *   q    [n_layers][B][Hq][D] bf16;  out [n_layers][B][Hq][D] bf16
 * One wave of CTAs cuts the (layer, request, KV head) x page work into equal
 * ranges (each (layer, request, KV head) weighs min(max_pages, block_topk+1)
 * pages, the selection size of a request with at least block_topk + 1
 * pages); a (layer, request, KV head) split between CTAs is merged by the
 * last of its pieces to finish, found by an atomic ticket.  ws is required:
 * it holds the partial softmax states and the tickets (zeroed before first
 * use, left zero by every call that completes).  SSA_ERR_INVALID_ARG when
 * ws is NULL.
 */
int ssa_sparse_paged_decode(const ssa_layout *lay, const ssa_cache *c, int layer0, int n_layers,
                            const void *q, const int32_t *sel, const int32_t *phys,
                            const int32_t *seq_lens, float sm_scale, void *out,
                            int32_t *status, void *ws, ssa_stream_t stream);

/*
 * Zero-copy host-tail attention (vLLM RFC #33980, the comment that maps one
 * address range with an HBM-backed head and a host-backed tail, so that the
 * attention reads the tail's slots over the interconnect with no staging
 * copy).  The same attention as ssa_sparse_paged_decode, on sel and the
 * block table instead of a remapped table: each selected page is resolved
 * through slot_of; a resident page is read from its pool slot, a page with
 * no slot straight from the pinned host mirror (16-byte loads over UVA into
 * the same on-chip layout).  The residency state is not changed -- no
 * ensure, no copy, no eviction -- so each step re-reads its host pages.
 *   sel          [n_layers][B][W] from ssa_index_topk
 *   block_table  [B][n_max] logical ids
 * Requires the host mirror (SSA_ERR_NO_MIRROR); ws as for
 * ssa_sparse_paged_decode.  Mirror bytes equal pool bytes, so the result is
 * that of ensure + remap + ssa_sparse_paged_decode on the same selection.
 */
int ssa_sparse_paged_decode_host_tail(const ssa_layout *lay, const ssa_cache *c, int layer0,
                                      int n_layers, const void *q, const int32_t *sel,
                                      const int32_t *block_table, const int32_t *seq_lens,
                                      float sm_scale, void *out, int32_t *status, void *ws,
                                      ssa_stream_t stream);

/*
 * ssa_index_topk without a workspace: the same indexer and top-k selection
 * (same arguments and results as ssa_index_topk, without scores_opt and ws),
 * for callers that cannot allocate device memory -- a plugin inside a host
 * program that owns every device allocation, or a serving loop that must not
 * allocate after start-up -- and so have no workspace to pass.
 *
 * The pages have no counterpart of this call; it only changes where the
 * score scratch lives.  That scratch is a fixed array of
 * SSA_STATIC_SCORE_ENTRIES int32 (4 MiB) compiled into the library, held on
 * every GPU that loads the library until the process exits.  A call needing
 * more than that (n_layers * batch * max_pages scores) returns
 * SSA_ERR_SCRATCH_LIMIT before enqueuing anything.  The call allocates and
 * frees nothing.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) and caches it: make that first call before
 * any stream capture.  Every call uses the same array, which keeps the last
 * call's scores; nothing in it needs clearing, but calls whose kernels
 * overlap on the GPU (other streams, other threads) race on it -- order them.
 */
#define SSA_STATIC_SCORE_ENTRIES (1u << 20)
int ssa_index_topk_static_scratch(const ssa_layout *lay, const ssa_cache *c, int layer0,
                                  int n_layers, const void *q, const int32_t *block_table,
                                  const int32_t *seq_lens, int32_t *sel, int32_t *n_sel,
                                  int32_t *status, ssa_stream_t stream);

/*
 * Failure-detection self-test (no counterpart in the pages): one CTA waits on
 * an mbarrier that nothing ever arrives on, using the bounded wait of every
 * kernel in this library (1 s of wall clock).  The wait gives up, the kernel
 * ORs SSA_ST_TIMEOUT into *status (device memory) and returns; the context
 * stays usable.  Takes about one second of GPU time.
 */
int ssa_selftest_bounded_wait(int32_t *status, ssa_stream_t stream);

/*
 * Measurement helper (no counterpart in the pages): the host link's rate for
 * reads issued by SMs, the access the miss fetch makes.  Copies n_chunks
 * chunks of chunk_bytes each, chunk i starting at byte offsets[i] of src,
 * into dst (chunk i at i * chunk_bytes), with 16-byte loads, loads_per_thread
 * (4, 8 or 16) in flight per thread, one group of 256-thread CTAs per chunk.
 *   src      pinned host memory the GPU can address (or device memory)
 *   dst      device memory, n_chunks * chunk_bytes bytes
 *   offsets  [n_chunks] int64, device memory; multiples of 16, and every
 *            chunk must lie inside the caller's source buffer (not checked:
 *            the values live on the device)
 * chunk_bytes a multiple of 16; 1 <= n_chunks <= 65535; src and dst 16-byte
 * aligned.  SSA_ERR_INVALID_ARG otherwise.  Time it with events on `stream`.
 */
int ssa_host_read_probe(const void *src, void *dst, const int64_t *offsets, int n_chunks,
                        int chunk_bytes, int loads_per_thread, ssa_stream_t stream);

/* Text for an SSA_ERR_* code or an SSA_ST_* bit set. */
const char *ssa_status_str(int code);

/* The cudaError_t of the last SSA_ERR_CUDA on this thread (0 if none). */
int ssa_last_cuda_error(void);

/* Number of kernel launches enqueued by calls on this thread so far. */
long long ssa_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* SSA_H */
