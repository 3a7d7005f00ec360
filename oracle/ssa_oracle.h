/*
 * ssa_oracle.h -- plain, slow CPU oracle for the sparse-attention decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path includes, links or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * Every function works on ONE layer.  Arrays are dense, row-major, and use the
 * same logical shapes as the library (the caller slices layers off):
 *   pool K/V codes   [S][Hkv][P][D]   (bf16 bit patterns, or e4m3 bytes)
 *   pool scales      [S][P]           fp32 (fp8 only)
 *   mirror K/V codes [Lp][Hkv][P][D], mirror scales [Lp][P]
 *   slab codes       [Lp][Hkv][D] int8, slab scale [Lp] fp32
 *   slab running sum [Lp][Hkv][D] fp32, slab count [Lp] int32
 *   slot_of [Lp], page_of [S], last_use [S], clock (scalar)
 * bf16 values travel as their uint16 bit patterns.
 *
 * parity pins: see tests/test_oracle_*.py (hand-worked example, hand LRU
 * trace, brute force, library routines, invariants).
 */
#ifndef SSA_ORACLE_H
#define SSA_ORACLE_H
#include <stdint.h>

typedef struct {
  int P;          /* tokens per page */
  int Hq, Hkv, D; /* query heads, KV heads, head dim */
  int fp8;        /* 0: bf16 K/V, 1: e4m3 codes with per-token fp32 scales */
  int Lp;         /* logical pages per layer */
  int S;          /* physical pool slots per layer */
  int B;          /* requests */
  int n_max;      /* block-table width (pages per request, max) */
  int k;          /* block_topk */
  int W;          /* max_sel_pages = 2k + 8 */
} or_layout;

/* --- number formats -------------------------------------------------- */
uint8_t or_e4m3_encode(float x);   /* round-to-nearest-even, saturating */
double  or_e4m3_decode(uint8_t c);
float   or_bf16_to_float(uint16_t b);

/* --- a0: store K/V through the write-through mirror, update the slab --- */
/* k, v: [T][Hkv][D] bf16 bits; pos: logical token ids (page*P + j).
 * mirror pointers may be NULL (no host tier).  Returns the number of tokens
 * whose page id was out of range (skipped). */
int or_store(const or_layout *L,
             uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
             uint8_t *k_mirror, uint8_t *v_mirror, float *k_scale_m, float *v_scale_m,
             int8_t *slab, float *slab_scale, float *slab_sum, int32_t *slab_cnt,
             const int32_t *slot_of,
             const uint16_t *k, const uint16_t *v, const int64_t *pos, int T);

/* --- a1: indexer scores ------------------------------------------------ */
/* q: [B][Hq][D] bf16 bits; bt: [B][n_max]; scores: [B][n_max] (entries at or
 * past a request's page count are INT32_MIN).  Returns #bad block-table ids. */
int or_index_scores(const or_layout *L, const int8_t *slab, const uint16_t *q,
                    const int32_t *bt, const int32_t *seq_lens, int32_t *scores);

/* --- a2: top-k page selection ----------------------------------------- */
/* sel: [B][W] ascending page indices (within the request), -1 padded;
 * n_sel: [B].  Returns the number of selected pages that did not fit W. */
int or_select(const or_layout *L, const int32_t *scores, const int32_t *seq_lens,
              int32_t *sel, int32_t *n_sel);

/* --- a3 + a4: LRU ensure, then copy misses mirror -> pool -------------- */
/* miss_page/miss_slot: [B*W], -1 padded.  *n_miss out.  Returns flags:
 * bit 1 = bad id, bit 2 = miss without a mirror, bit 3 = unresolved. */
int or_ensure(const or_layout *L, int32_t *slot_of, int32_t *page_of,
              int32_t *last_use, int32_t *clock,
              const int32_t *sel, const int32_t *bt,
              const uint8_t *k_mirror, const uint8_t *v_mirror,
              const float *k_scale_m, const float *v_scale_m,
              uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
              int32_t *miss_page, int32_t *miss_slot, int32_t *n_miss);

/* --- a5: logical -> physical remap ------------------------------------ */
/* phys: [B][W].  Returns the number of selected pages with no slot. */
int or_remap(const or_layout *L, const int32_t *slot_of, const int32_t *sel,
             const int32_t *bt, int32_t *phys);

/* --- a6 + a7: attention over the selected pages, exact, fp64 ---------- */
/* out: [B][Hq][D] doubles. */
void or_decode(const or_layout *L, const uint8_t *k_pool, const uint8_t *v_pool,
               const float *k_scale, const float *v_scale, const uint16_t *q,
               const int32_t *sel, const int32_t *phys, const int32_t *seq_lens,
               double sm_scale, double *out);

/* --- NEXT-2: one residency for the layers of a call -------------------- */
/* State: the first layer's arrays; sel [n_layers][B][W]; pools, scales and
 * mirrors: n_layers consecutive per-layer slices; miss lists [n_layers*B*W]. */
int or_ensure_shared(const or_layout *L, int n_layers, int32_t *slot_of, int32_t *page_of,
                     int32_t *last_use, int32_t *clock, const int32_t *sel, const int32_t *bt,
                     const uint8_t *k_mirror, const uint8_t *v_mirror,
                     const float *k_scale_m, const float *v_scale_m,
                     uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
                     int32_t *miss_page, int32_t *miss_slot, int32_t *n_miss);

/* --- NEXT-1: top-k preload after a step's ensure ---------------------- */
/* scores: [B][n_max] of the step (or_index_scores); 1 <= width <= W (else
 * -1).  miss lists [B*W] (-1 after n_miss).  Returns flags as or_ensure. */
int or_prefetch(const or_layout *L, int width, int32_t *slot_of, int32_t *page_of,
                int32_t *last_use, const int32_t *clock, const int32_t *scores,
                const int32_t *seq_lens, const int32_t *bt,
                const uint8_t *k_mirror, const uint8_t *v_mirror,
                const float *k_scale_m, const float *v_scale_m,
                uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
                int32_t *miss_page, int32_t *miss_slot, int32_t *n_miss);

/* --- threads ------------------------------------------------------------ */
/* Threads the independent loops may use (n <= 0: every core); results never
 * depend on it.  or_threads: the count now in force (1 without OpenMP). */
void or_set_threads(int n);
int or_threads(void);

#endif
