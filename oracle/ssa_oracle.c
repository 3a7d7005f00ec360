/*
 * ssa_oracle.c -- plain, slow CPU oracle for the per-layer
 * sparse-attention decode step: store through a write-through mirror, int8
 * indexer, top-k page selection, LRU ensure + miss copy, block-table remap,
 * exact attention over the selected pages.
 *
 * TEST INFRASTRUCTURE.  Only tests/, the smoke check and the benchmark's CPU
 * baseline use it; the CUDA library never does.  It shares no code with the
 * library.  Built with -O2 -ffp-contract=off and no fast-math, so every fp32
 * operation below is one correctly rounded IEEE operation in program order.
 * Loops whose iterations are independent (tokens of a store, pages of a
 * score, requests of a selection, (request, head) outputs of the attention)
 * carry OpenMP pragmas; each result is still computed by one thread in the
 * order written, so the results do not depend on the thread count, and
 * without OpenMP the pragmas are ignored.
 *
 * Sources (web pages, cited by title and section):
 *   [FT499]  FreeToken PR #499 "host-RAM KV tier for sparse-attention models
 *            (--kv-host-pages)": sections "What", "Why this works for sparse
 *            attention", "Design", "Known limitations".
 *   [FT525]  FreeToken PR #525 "host-resident prefix tier for hybrid GDN
 *            models", conversation summary (mirror_store_quant, scale banks,
 *            set_select_width).
 *   [RFC]    vLLM issue #33980 "[RFC]: Sparse attention KV cache offloading",
 *            "Proposed Change / KV cache management".
 * Where the pages leave a step open, the reading taken is stated at the step.
 */
#include "ssa_oracle.h"

#include <float.h>
#include <limits.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

float or_bf16_to_float(uint16_t b) {
  /* bf16 is the top half of an IEEE binary32. */
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* OCP 8-bit floating point, E4M3: 1 sign, 4 exponent bits (bias 7), 3
 * mantissa bits; no infinities; S.1111.111 is NaN, so the largest finite
 * magnitude is 1.75 * 2^8 = 448.  Exponent field 0 holds subnormals
 * m * 2^-9.  Encoding rounds to nearest, ties to even, and saturates to
 * +-448 (the fp8 KV cache stores finite codes only). */
double or_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9);
  else
    mag = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

uint8_t or_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E; /* saturate: 0 1111 110 = 448 */
  /* Spacing of representable values next to a: 2^(e-3) inside binade
   * [2^e, 2^(e+1)) for e >= -6; subnormals share the spacing 2^-9. */
  int ex;
  frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) -> binade exponent ex-1 */
  int be = ex - 1;
  if (a == 0.0 || be < -6) be = -6;
  double quantum = ldexp(1.0, be - 3);
  double r = nearbyint(a / quantum) * quantum; /* exact scaling, RNE */
  if (r > 448.0) r = 448.0;                    /* cannot happen below 448 */
  if (r == 0.0) return sign;
  if (r < ldexp(1.0, -6)) { /* subnormal: r = m * 2^-9, m in 1..7 */
    int m = (int)(r / ldexp(1.0, -9));
    return sign | (uint8_t)m;
  }
  frexp(r, &ex);
  int e = ex - 1;                                     /* r in [2^e, 2^(e+1)) */
  int m = (int)((r / ldexp(1.0, e) - 1.0) * 8.0);     /* exact */
  return sign | (uint8_t)(((e + 7) << 3) | m);
}

/* ------------------------------------------------------------------------ */
/* a0: store, write-through mirror, slab                                     */
/* ------------------------------------------------------------------------ */

static size_t page_elems(const or_layout *L) { return (size_t)L->Hkv * L->P * L->D; }

/* Element (h, j, d) of a page block [Hkv][P][D]. */
static size_t in_page(const or_layout *L, int h, int j, int d) {
  return ((size_t)h * L->P + j) * L->D + d;
}

/*
 * [FT499] "Design": each stored token also goes to pinned host memory, so a
 * slot can be evicted without a write-back.  [FT525]: with fp8 that host copy
 * gets the quantised codes and their scales, so mirror and pool hold the same
 * bytes.
 *
 * fp8 reading (per-token scale, [FT525] "the fp8 pool's per-token
 * _scale_buffer"): one fp32 scale per token per tensor over all KV heads,
 * s = amax/448 (s = 1 when amax = 0); code = e4m3(x / s).
 *
 * Slab reading ([FT499] "Why this works": the indexer runs over a compressed,
 * GPU-resident slab): per logical page, the fp32 sum of the stored bf16 keys
 * accumulated in token order, mean = sum / count, one symmetric int8 scale per
 * page over all heads, s = amax|mean| / 127, code = clamp(rint(mean / s)).
 */
int or_store(const or_layout *L,
             uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
             uint8_t *k_mirror, uint8_t *v_mirror, float *k_scale_m, float *v_scale_m,
             int8_t *slab, float *slab_scale, float *slab_sum, int32_t *slab_cnt,
             const int32_t *slot_of,
             const uint16_t *k, const uint16_t *v, const int64_t *pos, int T) {
  const int HD = L->Hkv * L->D;
  const size_t esz = L->fp8 ? 1 : 2;
  int bad = 0;
  /* 1. each token's codes (and scale) into the mirror and, when resident, the
   *    slot.  Tokens write disjoint bytes (positions are distinct), so the
   *    loop runs its iterations in any order. */
#pragma omp parallel for schedule(static) reduction(+ : bad)
  for (int t = 0; t < T; ++t) {
    int64_t page64 = pos[t] / L->P;
    if (pos[t] < 0 || page64 >= L->Lp) { ++bad; continue; }
    int page = (int)page64, j = (int)(pos[t] % L->P);
    int slot = slot_of[page];
    for (int which = 0; which < 2; ++which) {
      const uint16_t *x = (which ? v : k) + (size_t)t * HD;
      uint8_t *pool = which ? v_pool : k_pool;
      uint8_t *mirror = which ? v_mirror : k_mirror;
      float *psc = which ? v_scale : k_scale;
      float *msc = which ? v_scale_m : k_scale_m;
      float s = 1.0f;
      if (L->fp8) {
        float amax = 0.0f;
        for (int i = 0; i < HD; ++i) {
          float a = fabsf(or_bf16_to_float(x[i]));
          if (a > amax) amax = a;
        }
        s = amax > 0.0f ? amax / 448.0f : 1.0f;
      }
      for (int h = 0; h < L->Hkv; ++h)
        for (int d = 0; d < L->D; ++d) {
          uint16_t xb = x[h * L->D + d];
          size_t off = in_page(L, h, j, d) * esz;
          uint8_t code8 = 0;
          if (L->fp8) code8 = or_e4m3_encode(or_bf16_to_float(xb) / s);
          if (mirror) {
            uint8_t *m = mirror + (size_t)page * page_elems(L) * esz + off;
            if (L->fp8) m[0] = code8; else memcpy(m, &xb, 2);
          }
          if (slot >= 0) {
            uint8_t *p = pool + (size_t)slot * page_elems(L) * esz + off;
            if (L->fp8) p[0] = code8; else memcpy(p, &xb, 2);
          }
        }
      if (L->fp8) {
        if (msc) msc[(size_t)page * L->P + j] = s;
        if (slot >= 0) psc[(size_t)slot * L->P + j] = s;
      }
    }
  }
  /* 2. slab running sums, in token order within each page.  With positions
   *    increasing (the store contract) a page's tokens form one contiguous
   *    run of the call: runs are independent and each is summed front to
   *    back.  Otherwise every token is summed in call order, one by one. */
  int *run0 = (int *)malloc(sizeof(int) * ((size_t)T + 1));
  int nrun = 0, ordered = 1;
  int64_t prev = -1;
  for (int t = 0; t < T; ++t) {
    if (pos[t] < 0 || pos[t] / L->P >= L->Lp) continue;
    if (pos[t] <= prev) ordered = 0;
    prev = pos[t];
    if (nrun == 0 || pos[t] / L->P != pos[run0[nrun - 1]] / L->P) run0[nrun++] = t;
  }
  char *touched = (char *)calloc((size_t)L->Lp, 1);
  if (ordered) {
#pragma omp parallel for schedule(dynamic, 64)
    for (int r = 0; r < nrun; ++r) {
      const int64_t page = pos[run0[r]] / L->P;
      float *sum = slab_sum + (size_t)page * HD;
      const int t1 = r + 1 < nrun ? run0[r + 1] : T;
      for (int t = run0[r]; t < t1; ++t) {
        if (pos[t] < 0 || pos[t] / L->P != page) continue;   /* out-of-range ids */
        const uint16_t *xk = k + (size_t)t * HD;
        for (int i = 0; i < HD; ++i) sum[i] = sum[i] + or_bf16_to_float(xk[i]);
        slab_cnt[page] += 1;
      }
      touched[page] = 1;
    }
  } else {
    for (int t = 0; t < T; ++t) {
      if (pos[t] < 0 || pos[t] / L->P >= L->Lp) continue;
      const int64_t page = pos[t] / L->P;
      const uint16_t *xk = k + (size_t)t * HD;
      float *sum = slab_sum + (size_t)page * HD;
      for (int i = 0; i < HD; ++i) sum[i] = sum[i] + or_bf16_to_float(xk[i]);
      slab_cnt[page] += 1;
      touched[page] = 1;
    }
  }
  free(run0);
  /* 3. re-quantise every page this call touched (pages are independent) */
#pragma omp parallel
  {
    float *mean = (float *)malloc(sizeof(float) * HD);
#pragma omp for schedule(dynamic, 256)
    for (int page = 0; page < L->Lp; ++page) {
      if (!touched[page]) continue;
      const float *sum = slab_sum + (size_t)page * HD;
      float cnt = (float)slab_cnt[page];
      float amax = 0.0f;
      for (int i = 0; i < HD; ++i) {
        mean[i] = sum[i] / cnt;
        if (fabsf(mean[i]) > amax) amax = fabsf(mean[i]);
      }
      float s = amax / 127.0f;
      slab_scale[page] = s;
      for (int i = 0; i < HD; ++i) {
        int c = 0;
        if (amax > 0.0f) {
          float r = rintf(mean[i] / s);
          c = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int)r);
        }
        slab[(size_t)page * HD + i] = (int8_t)c;
      }
    }
    free(mean);
  }
  free(touched);
  return bad;
}

/* ------------------------------------------------------------------------ */
/* a1: indexer score                                                         */
/* ------------------------------------------------------------------------ */

static int pages_of(const or_layout *L, int seq_len) {
  int n = (seq_len + L->P - 1) / L->P;
  return n > L->n_max ? L->n_max : (n < 0 ? 0 : n);
}

/*
 * [FT499] "Why this works": the indexer scores every page from the compressed
 * slab before any page is read.  Reading: q is quantised to int8 with one
 * symmetric scale per request over all query heads (s = amax|q|/127), and the
 * page score is the exact integer
 *     S[b, p] = sum_hq sum_d q8[b, hq, d] * k8[bt[b, p], hq / G, d],
 * query head hq reading KV head hq / G (contiguous groups of G = Hq / Hkv).
 * The int32 sum alone ranks pages; the page scale does not weight it.
 */
int or_index_scores(const or_layout *L, const int8_t *slab, const uint16_t *q,
                    const int32_t *bt, const int32_t *seq_lens, int32_t *scores) {
  const int G = L->Hq / L->Hkv, HQD = L->Hq * L->D;
  int bad = 0;
  int32_t *q8 = (int32_t *)malloc(sizeof(int32_t) * (size_t)L->B * HQD);
  for (int b = 0; b < L->B; ++b) {
    const uint16_t *qb = q + (size_t)b * HQD;
    int32_t *q8b = q8 + (size_t)b * HQD;
    float amax = 0.0f;
    for (int i = 0; i < HQD; ++i) {
      float a = fabsf(or_bf16_to_float(qb[i]));
      if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    for (int i = 0; i < HQD; ++i) {
      int c = 0;
      if (amax > 0.0f) {
        float r = rintf(or_bf16_to_float(qb[i]) / s);
        c = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int)r);
      }
      q8b[i] = c;
    }
  }
  /* every score is its own exact integer sum: pages in any order */
  const long long total = (long long)L->B * L->n_max;
#pragma omp parallel for schedule(static) reduction(+ : bad)
  for (long long bp = 0; bp < total; ++bp) {
    const int b = (int)(bp / L->n_max), p = (int)(bp % L->n_max);
    const int32_t *q8b = q8 + (size_t)b * HQD;
    int32_t *out = &scores[bp];
    *out = INT32_MIN;
    if (p >= pages_of(L, seq_lens[b])) continue;
    int id = bt[(size_t)b * L->n_max + p];
    if (id < 0 || id >= L->Lp) { ++bad; continue; }
    int64_t acc = 0;
    for (int hq = 0; hq < L->Hq; ++hq)
      for (int d = 0; d < L->D; ++d)
        acc += (int64_t)q8b[hq * L->D + d] *
               (int64_t)slab[((size_t)id * L->Hkv + hq / G) * L->D + d];
    *out = (int32_t)acc;
  }
  free(q8);
  return bad;
}

/* ------------------------------------------------------------------------ */
/* a2: top-k selection                                                       */
/* ------------------------------------------------------------------------ */

typedef struct { int32_t score; int32_t page; } cand;

/* Higher score first; equal scores: lower page id first. */
static int cand_cmp(const void *a, const void *b) {
  const cand *x = (const cand *)a, *y = (const cand *)b;
  if (x->score != y->score) return x->score > y->score ? -1 : 1;
  return x->page < y->page ? -1 : (x->page > y->page);
}

static int int_cmp(const void *a, const void *b) {
  int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
  return x < y ? -1 : (x > y);
}

/*
 * [FT499] "Why this works" (top-k block selection over the slab, fixed shape)
 * and "Design" (compact_selected_pages with a drop counter; max_sel_pages =
 * 2*block_topk + 8).  Reading: the k best pages among [0, n-1) by (score
 * desc, page id asc), plus the last page n-1 always; all pages when n-1 <= k.
 * The list is written in ascending page order and padded with -1 to W; pages
 * that would not fit W are counted as drops.
 */
int or_select(const or_layout *L, const int32_t *scores, const int32_t *seq_lens,
              int32_t *sel, int32_t *n_sel) {
  int drops = 0;
#pragma omp parallel reduction(+ : drops)
  {
    cand *c = (cand *)malloc(sizeof(cand) * (L->n_max + 1));
    int32_t *chosen = (int32_t *)malloc(sizeof(int32_t) * (L->n_max + 1));
#pragma omp for schedule(dynamic, 1)
    for (int b = 0; b < L->B; ++b) {
      int n = pages_of(L, seq_lens[b]);
      int m = 0;
      if (n > 0) {
        if (n - 1 <= L->k) {
          for (int p = 0; p < n; ++p) chosen[m++] = p;
        } else {
          for (int p = 0; p < n - 1; ++p) {
            c[p].score = scores[(size_t)b * L->n_max + p];
            c[p].page = p;
          }
          qsort(c, (size_t)(n - 1), sizeof(cand), cand_cmp);
          for (int i = 0; i < L->k; ++i) chosen[m++] = c[i].page;
          chosen[m++] = n - 1;
          qsort(chosen, (size_t)m, sizeof(int32_t), int_cmp);
        }
      }
      int kept = m < L->W ? m : L->W;
      drops += m - kept;
      for (int i = 0; i < L->W; ++i)
        sel[(size_t)b * L->W + i] = i < kept ? chosen[i] : -1;
      n_sel[b] = kept;
    }
    free(chosen);
    free(c);
  }
  return drops;
}

/* ------------------------------------------------------------------------ */
/* a3 + a4: LRU ensure and miss copy                                          */
/* ------------------------------------------------------------------------ */

typedef struct { int32_t key; int32_t slot; } victim;

static int victim_cmp(const void *a, const void *b) {
  const victim *x = (const victim *)a, *y = (const victim *)b;
  if (x->key != y->key) return x->key < y->key ? -1 : 1;
  return x->slot < y->slot ? -1 : (x->slot > y->slot);
}

/*
 * [FT499] "What" and "Design": the GPU's slots cache logical pages, the
 * least recently used slot is reused first, the update has fixed shapes, and
 * evicting only rebinds a slot (the host copy is always current, so nothing
 * is written back); misses are copied from the pinned host copy; [FT525]: the
 * copy includes the fp8 scales, and the pool is sized so that the batch's
 * whole selection fits.
 *
 * Reading of the order of events (the pages state none):
 *   1. U = the distinct logical ids selected by the batch, ascending.
 *   2. hits (slot_of >= 0) are touched: last_use = clock.
 *   3. misses take victims in order: free slots by ascending slot id, then
 *      bound slots not touched this step by ascending (last_use, slot).
 *   4. the i-th miss (ascending id) is bound to the i-th victim; the victim's
 *      old page loses its slot; the page data is copied mirror -> slot.
 *   5. clock += 1.
 */
int or_ensure(const or_layout *L, int32_t *slot_of, int32_t *page_of,
              int32_t *last_use, int32_t *clock,
              const int32_t *sel, const int32_t *bt,
              const uint8_t *k_mirror, const uint8_t *v_mirror,
              const float *k_scale_m, const float *v_scale_m,
              uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
              int32_t *miss_page, int32_t *miss_slot, int32_t *n_miss) {
  int flags = 0;
  const int BW = L->B * L->W;
  const int32_t now = *clock;
  int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (BW + 1));
  int nid = 0;
  for (int b = 0; b < L->B; ++b)
    for (int i = 0; i < L->W; ++i) {
      int p = sel[(size_t)b * L->W + i];
      if (p < 0) continue;
      if (p >= L->n_max) { flags |= 2; continue; }
      int id = bt[(size_t)b * L->n_max + p];
      if (id < 0 || id >= L->Lp) { flags |= 2; continue; }
      ids[nid++] = id;
    }
  qsort(ids, (size_t)nid, sizeof(int32_t), int_cmp);
  int nu = 0;
  for (int i = 0; i < nid; ++i)
    if (nu == 0 || ids[nu - 1] != ids[i]) ids[nu++] = ids[i];

  /* 2: touch hits */
  for (int i = 0; i < nu; ++i)
    if (slot_of[ids[i]] >= 0) last_use[slot_of[ids[i]]] = now;

  /* 3: victim order */
  victim *cands = (victim *)malloc(sizeof(victim) * (L->S + 1));
  int nc = 0;
  for (int s = 0; s < L->S; ++s) {
    if (page_of[s] >= 0 && last_use[s] == now) continue; /* touched: a hit */
    cands[nc].key = page_of[s] < 0 ? -2 : last_use[s];
    cands[nc].slot = s;
    ++nc;
  }
  qsort(cands, (size_t)nc, sizeof(victim), victim_cmp);

  /* 4: bind misses, copy */
  const size_t esz = L->fp8 ? 1 : 2;
  const size_t pbytes = page_elems(L) * esz;
  int m = 0;
  for (int i = 0; i < nu; ++i) {
    int id = ids[i];
    if (slot_of[id] >= 0) continue;
    if (m >= nc) { flags |= 8; continue; } /* pool too small: unresolved */
    int v = cands[m].slot;
    int old = page_of[v];
    if (old >= 0) slot_of[old] = -1;
    slot_of[id] = v;
    page_of[v] = id;
    last_use[v] = now;
    if (k_mirror && v_mirror) {
      memcpy(k_pool + (size_t)v * pbytes, k_mirror + (size_t)id * pbytes, pbytes);
      memcpy(v_pool + (size_t)v * pbytes, v_mirror + (size_t)id * pbytes, pbytes);
      if (L->fp8) {
        memcpy(k_scale + (size_t)v * L->P, k_scale_m + (size_t)id * L->P, sizeof(float) * L->P);
        memcpy(v_scale + (size_t)v * L->P, v_scale_m + (size_t)id * L->P, sizeof(float) * L->P);
      }
    } else {
      flags |= 4;
    }
    miss_page[m] = id;
    miss_slot[m] = v;
    ++m;
  }
  for (int i = m; i < BW; ++i) miss_page[i] = miss_slot[i] = -1;
  *n_miss = m;
  *clock = now + 1;
  free(cands);
  free(ids);
  return flags;
}

/* ------------------------------------------------------------------------ */
/* NEXT-2: residency shared by the layers of a call                           */
/* ------------------------------------------------------------------------ */

/*
 * [FT499] "Design", residency engine bullet: one launch copies a page's K and
 * V for all the sparse-attention layers, i.e. a logical page is resident (or
 * not) for every layer at once.  Reading: for a call over layers
 * [0, n_layers) (the arrays below are those layers' consecutive slices), one
 * LRU state -- the first layer's slot_of / page_of / last_use / clock -- is
 * shared; the ensure works on the union of every layer's selection with the
 * order of events of or_ensure (distinct ids ascending, hits touched, misses
 * ascending take victims, clock + 1), and each miss is copied mirror -> slot
 * for every layer.  The other layers' LRU arrays are not used.  The state
 * update is exactly or_ensure on the layers' selections stacked as one batch
 * of n_layers * B requests; the copy then repeats for layers 1..n-1.
 *   sel [n_layers][B][W]; pools and mirrors: [n_layers] slices of the
 *   per-layer layouts; miss lists [n_layers * B * W].
 */
int or_ensure_shared(const or_layout *L, int n_layers, int32_t *slot_of, int32_t *page_of,
                     int32_t *last_use, int32_t *clock, const int32_t *sel, const int32_t *bt,
                     const uint8_t *k_mirror, const uint8_t *v_mirror,
                     const float *k_scale_m, const float *v_scale_m,
                     uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
                     int32_t *miss_page, int32_t *miss_slot, int32_t *n_miss) {
  or_layout Lu = *L;
  Lu.B = L->B * n_layers;
  int32_t *btu = (int32_t *)malloc(sizeof(int32_t) * (size_t)Lu.B * L->n_max);
  for (int l = 0; l < n_layers; ++l)
    memcpy(btu + (size_t)l * L->B * L->n_max, bt, sizeof(int32_t) * (size_t)L->B * L->n_max);
  const size_t esz = L->fp8 ? 1 : 2;
  const size_t pbytes = page_elems(L) * esz;
  const size_t mirror_layer = (size_t)L->Lp * pbytes, pool_layer = (size_t)L->S * pbytes;
  int flags = or_ensure(&Lu, slot_of, page_of, last_use, clock, sel, btu,
                        k_mirror, v_mirror, k_scale_m, v_scale_m,
                        k_pool, v_pool, k_scale, v_scale, miss_page, miss_slot, n_miss);
  for (int l = 1; l < n_layers; ++l)
    for (int i = 0; i < *n_miss; ++i) {
      const int id = miss_page[i], v = miss_slot[i];
      if (!(k_mirror && v_mirror)) continue;
      memcpy(k_pool + l * pool_layer + (size_t)v * pbytes,
             k_mirror + l * mirror_layer + (size_t)id * pbytes, pbytes);
      memcpy(v_pool + l * pool_layer + (size_t)v * pbytes,
             v_mirror + l * mirror_layer + (size_t)id * pbytes, pbytes);
      if (L->fp8) {
        memcpy(k_scale + ((size_t)l * L->S + v) * L->P, k_scale_m + ((size_t)l * L->Lp + id) * L->P,
               sizeof(float) * L->P);
        memcpy(v_scale + ((size_t)l * L->S + v) * L->P, v_scale_m + ((size_t)l * L->Lp + id) * L->P,
               sizeof(float) * L->P);
      }
    }
  free(btu);
  return flags;
}

/* ------------------------------------------------------------------------ */
/* NEXT-1: top-k preload                                                      */
/* ------------------------------------------------------------------------ */

/*
 * [RFC] "Motivation" point 2 and "Proposed Change / Topk KV preload": the
 * top-k of adjacent decode steps overlap strongly, so a former top-k index can
 * drive a fetch that runs while the current step computes, and only the pages
 * still missing once the actual top-k is known are loaded synchronously.
 *
 * Reading (the pages give no rule; this one keeps the fixed shapes and the
 * LRU above):
 *   * it runs after a step's ensure, on that step's scores; e = clock - 1 is
 *     the epoch of that ensure (its pages have last_use == e);
 *   * candidates, per request: the top (width - 1) pages of [0, n-1) by
 *     (score desc, page id asc) plus page n-1, all pages when n-1 <= width-1
 *     (the selection of or_select with k = width - 1), width <= W;
 *   * U = the distinct logical ids of the batch's candidates, ascending;
 *   * resident ids of U are touched: last_use = e, as the step's own pages
 *     are, so that the preload never evicts a candidate;
 *   * the ids of U that are not resident, ascending, take victims in order:
 *     free slots by ascending slot id, then bound slots with last_use < e by
 *     ascending (last_use, slot) -- the pages the current step reads and
 *     the candidates are never evicted; ids left over when the victims run
 *     out are not fetched;
 *   * each bound id gets last_use = e, its slot the mirror's bytes;
 *   * the clock does not move, so the next ensure sees the preloaded pages
 *     as resident (hits) and, among the slots its own step does not touch,
 *     evicts the least recently used first.
 */
int or_prefetch(const or_layout *L, int width, int32_t *slot_of, int32_t *page_of,
                int32_t *last_use, const int32_t *clock, const int32_t *scores,
                const int32_t *seq_lens, const int32_t *bt,
                const uint8_t *k_mirror, const uint8_t *v_mirror,
                const float *k_scale_m, const float *v_scale_m,
                uint8_t *k_pool, uint8_t *v_pool, float *k_scale, float *v_scale,
                int32_t *miss_page, int32_t *miss_slot, int32_t *n_miss) {
  int flags = 0;
  const int BW = L->B * L->W;
  const int32_t e = *clock - 1;
  if (width < 1 || width > L->W) return -1;
  or_layout Lw = *L;
  Lw.k = width - 1;
  Lw.W = width;
  int32_t *cand = (int32_t *)malloc(sizeof(int32_t) * (size_t)L->B * width);
  int32_t *ncand = (int32_t *)malloc(sizeof(int32_t) * L->B);
  or_select(&Lw, scores, seq_lens, cand, ncand);

  int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * ((size_t)L->B * width + 1));
  int nid = 0;
  for (int b = 0; b < L->B; ++b)
    for (int i = 0; i < ncand[b]; ++i) {
      int p = cand[(size_t)b * width + i];
      int id = bt[(size_t)b * L->n_max + p];
      if (id < 0 || id >= L->Lp) { flags |= 2; continue; }
      ids[nid++] = id;
    }
  qsort(ids, (size_t)nid, sizeof(int32_t), int_cmp);
  int nu = 0;
  for (int i = 0; i < nid; ++i)
    if (nu == 0 || ids[nu - 1] != ids[i]) ids[nu++] = ids[i];

  /* touch the resident candidates */
  for (int i = 0; i < nu; ++i)
    if (slot_of[ids[i]] >= 0) last_use[slot_of[ids[i]]] = e;

  /* victim order: free slots, then bound slots older than epoch e */
  victim *cands = (victim *)malloc(sizeof(victim) * (L->S + 1));
  int nc = 0;
  for (int s = 0; s < L->S; ++s) {
    if (page_of[s] >= 0 && last_use[s] >= e) continue;
    cands[nc].key = page_of[s] < 0 ? -2 : last_use[s];
    cands[nc].slot = s;
    ++nc;
  }
  qsort(cands, (size_t)nc, sizeof(victim), victim_cmp);

  const size_t esz = L->fp8 ? 1 : 2;
  const size_t pbytes = page_elems(L) * esz;
  int m = 0;
  for (int i = 0; i < nu && m < nc; ++i) {
    int id = ids[i];
    if (slot_of[id] >= 0) continue;
    int v = cands[m].slot;
    int old = page_of[v];
    if (old >= 0) slot_of[old] = -1;
    slot_of[id] = v;
    page_of[v] = id;
    last_use[v] = e;
    if (k_mirror && v_mirror) {
      memcpy(k_pool + (size_t)v * pbytes, k_mirror + (size_t)id * pbytes, pbytes);
      memcpy(v_pool + (size_t)v * pbytes, v_mirror + (size_t)id * pbytes, pbytes);
      if (L->fp8) {
        memcpy(k_scale + (size_t)v * L->P, k_scale_m + (size_t)id * L->P, sizeof(float) * L->P);
        memcpy(v_scale + (size_t)v * L->P, v_scale_m + (size_t)id * L->P, sizeof(float) * L->P);
      }
    } else {
      flags |= 4;
    }
    miss_page[m] = id;
    miss_slot[m] = v;
    ++m;
  }
  for (int i = m; i < BW; ++i) miss_page[i] = miss_slot[i] = -1;
  *n_miss = m;
  free(cands);
  free(ids);
  free(ncand);
  free(cand);
  return flags;
}

/* ------------------------------------------------------------------------ */
/* a5: remap                                                                 */
/* ------------------------------------------------------------------------ */

/* [FT499] "Design": after ensure, the block table is translated from logical
 * to physical ids and the attention kernel runs on it unmodified. */
int or_remap(const or_layout *L, const int32_t *slot_of, const int32_t *sel,
             const int32_t *bt, int32_t *phys) {
  int unresolved = 0;
  for (int b = 0; b < L->B; ++b)
    for (int i = 0; i < L->W; ++i) {
      int p = sel[(size_t)b * L->W + i];
      int out = -1;
      if (p >= 0) {
        int id = (p < L->n_max) ? bt[(size_t)b * L->n_max + p] : -1;
        if (id >= 0 && id < L->Lp) out = slot_of[id];
        if (out < 0) ++unresolved;
      }
      phys[(size_t)b * L->W + i] = out;
    }
  return unresolved;
}

/* ------------------------------------------------------------------------ */
/* a6 + a7: attention over the selected pages                                */
/* ------------------------------------------------------------------------ */

/*
 * [FT499] "Design": the sparse paged attention reads only the selected pages
 * through the remapped table.  This is the exact definition, in fp64, on the
 * values the pool holds (bf16 values, or e4m3 code * per-token scale):
 *   o[b, hq] = sum_t softmax_t(sm_scale * q[b, hq] . K[t]) V[t]
 * over the tokens t = p*P + j of the selected pages p with t < seq_len[b],
 * read from KV head hq / G.  Split-and-merge is an implementation choice and
 * does not appear here.
 */
void or_decode(const or_layout *L, const uint8_t *k_pool, const uint8_t *v_pool,
               const float *k_scale, const float *v_scale, const uint16_t *q,
               const int32_t *sel, const int32_t *phys, const int32_t *seq_lens,
               double sm_scale, double *out) {
  const int G = L->Hq / L->Hkv, D = L->D;
  const size_t esz = L->fp8 ? 1 : 2;
  const size_t ntok_max = (size_t)L->W * L->P;
  /* the token list of every request: (slot, row) pairs in selection order */
  int32_t *tslot = (int32_t *)malloc(sizeof(int32_t) * ntok_max * L->B);
  int32_t *tj = (int32_t *)malloc(sizeof(int32_t) * ntok_max * L->B);
  size_t *ntok = (size_t *)malloc(sizeof(size_t) * L->B);
  for (int b = 0; b < L->B; ++b) {
    size_t nt = 0;
    for (int i = 0; i < L->W; ++i) {
      int p = sel[(size_t)b * L->W + i], s = phys[(size_t)b * L->W + i];
      if (p < 0 || s < 0) continue;
      for (int j = 0; j < L->P; ++j) {
        if ((int64_t)p * L->P + j >= seq_lens[b]) break;
        tslot[b * ntok_max + nt] = s;
        tj[b * ntok_max + nt] = j;
        ++nt;
      }
    }
    ntok[b] = nt;
  }
  /* every (request, query head) output is computed whole by one thread */
#pragma omp parallel
  {
    double *sc = (double *)malloc(sizeof(double) * (ntok_max + 1));
    double *qd = (double *)malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 1)
    for (int bh = 0; bh < L->B * L->Hq; ++bh) {
      const int b = bh / L->Hq, hq = bh % L->Hq;
      const int h = hq / G;
      const size_t nt = ntok[b];
      const int32_t *ts = tslot + b * ntok_max, *tjj = tj + b * ntok_max;
      double *o = out + ((size_t)b * L->Hq + hq) * D;
      for (int d = 0; d < D; ++d) {
        qd[d] = or_bf16_to_float(q[((size_t)b * L->Hq + hq) * D + d]);
        o[d] = 0.0;
      }
      if (nt == 0) continue;
      double mx = -INFINITY;
      for (size_t t = 0; t < nt; ++t) {
        size_t base = ((size_t)ts[t] * L->Hkv + h) * L->P + tjj[t];
        double dot = 0.0;
        for (int d = 0; d < D; ++d) {
          double kv;
          if (L->fp8) {
            kv = or_e4m3_decode(k_pool[base * D + d]) *
                 (double)k_scale[(size_t)ts[t] * L->P + tjj[t]];
          } else {
            uint16_t bits;
            memcpy(&bits, k_pool + (base * D + d) * esz, 2);
            kv = or_bf16_to_float(bits);
          }
          dot += qd[d] * kv;
        }
        sc[t] = sm_scale * dot;
        if (sc[t] > mx) mx = sc[t];
      }
      double l = 0.0;
      for (size_t t = 0; t < nt; ++t) {
        double w = exp(sc[t] - mx);
        l += w;
        size_t base = ((size_t)ts[t] * L->Hkv + h) * L->P + tjj[t];
        for (int d = 0; d < D; ++d) {
          double vv;
          if (L->fp8) {
            vv = or_e4m3_decode(v_pool[base * D + d]) *
                 (double)v_scale[(size_t)ts[t] * L->P + tjj[t]];
          } else {
            uint16_t bits;
            memcpy(&bits, v_pool + (base * D + d) * esz, 2);
            vv = or_bf16_to_float(bits);
          }
          o[d] += w * vv;
        }
      }
      for (int d = 0; d < D; ++d) o[d] /= l;
    }
    free(qd);
    free(sc);
  }
  free(ntok);
  free(tj);
  free(tslot);
}

/* Threads the parallel loops above may use (<= 0: the OpenMP default, every
 * core).  Results do not depend on it: each output element is computed by
 * one thread in a fixed order. */
void or_set_threads(int n) {
#ifdef _OPENMP
  omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
  (void)n;
#endif
}

int or_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
