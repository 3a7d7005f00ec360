// index.cu -- a1 indexer scores and a2 top-k page selection.
//
// FreeToken PR #499, "Why this works for sparse attention": every attend step
// first runs top-k block selection over a compressed, GPU-resident slab, and
// only then reads the selected pages; the selection has a fixed shape.
// "Design": the compacted selection counts drops; its width is
// max_sel_pages = 2*block_topk + 8.
//
// Score (exact integer arithmetic, so any summation order gives the same
// int32):  S[b,p] = sum_hq sum_d q8[b,hq,d] * slab[bt[b,p], hq/G, d].
// The G query heads of one KV head are summed first (|sum| <= 127*G fits
// int16), then dotted with the page's int8 codes by __dp2a (16-bit x 8-bit).
// The slab scan is an HBM stream: a GEMV, not a dense contraction, so it runs
// on the integer ALUs with 16-byte coalesced loads, not on tensor cores.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace ssa {
namespace {

constexpr int kScoreThreads = 256;
constexpr int kScoreIters = 8;     // pages per lane group per round (loads in flight)

struct ScoreParams {
  const int8_t* slab;              // [Lyr][Lp][HD]
  const __nv_bfloat16* q;          // [n_layers][B][Hq][D]
  const int32_t* bt;               // [B][nmax]
  const int32_t* seq_lens;         // [B]
  int32_t* scores;                 // [n_layers][B][nmax]
  int32_t* status;
  int layer0, Lp, B, Hq, Hkv, G, D, P, nmax;
  int lanes;                       // lanes per page (power of two <= 32)
  int pages_per_cta;
};

// Scores of this CTA's chunk of pages of request blockIdx.y, layer blockIdx.z.
// CPL: 16-byte chunks per lane (HD = 16 * lanes * CPL).  qg: [Hkv][D] int16
// shared memory for the group sums of q8.
template <int CPL>
__device__ __forceinline__ void score_chunk(const ScoreParams& p, int16_t* qg, int8_t* q8s,
                                            float* red) {
  const int li = blockIdx.z, b = blockIdx.y;
  const int HD = p.Hkv * p.D;
  const int L = p.lanes;
  const int sub = threadIdx.x & (L - 1), grp = threadIdx.x / L;
  const int groups = blockDim.x / L;
  const int p0 = blockIdx.x * p.pages_per_cta;
  const int p1 = min(p.nmax, p0 + p.pages_per_cta);
  const int n_b = min(p.nmax, (p.seq_lens[b] + p.P - 1) / p.P);
  const int8_t* slab_l = p.slab + (size_t)(p.layer0 + li) * p.Lp * HD;
  int32_t* out = p.scores + ((size_t)li * p.B + b) * p.nmax;

  // 1. loads that depend on nothing go out first: q (16-byte vectors, the
  //    whole [Hq][D] row of the request spread over the CTA) and the
  //    block-table ids of the first round of pages
  const __nv_bfloat16* qb = p.q + ((size_t)li * p.B + b) * p.Hq * p.D;
  const int nq16 = p.Hq * p.D / 8;               // 16-byte vectors of q
  constexpr int kQV = 4;                          // Hq * D <= 8 * 4 * 256
  uint4 qraw[kQV];
#pragma unroll
  for (int j = 0; j < kQV; ++j) {
    const int i = threadIdx.x + j * blockDim.x;
    qraw[j] = i < nq16 ? reinterpret_cast<const uint4*>(qb)[i] : make_uint4(0, 0, 0, 0);
  }
  int4 v[kScoreIters][CPL];
  bool live[kScoreIters];          // a slab row was loaded (the id is in range)
  // a round's block-table ids: lane sub < kScoreIters of each page group
  // loads the id of the group's page sub of the round (one register), and
  // the round's loads take them by shuffles within the group; the next
  // round's ids are loaded while this round is scored
  static_assert(kScoreIters <= 8, "the lanes of a page group hold a round's ids");
  int id_lane = -1;
  auto load_ids = [&](int base) {
    const int pg = base + (sub & (kScoreIters - 1)) * groups + grp;
    id_lane = sub < kScoreIters && pg < p1 ? p.bt[(size_t)b * p.nmax + pg] : -1;
  };
  int ids[kScoreIters];
  // the slab loads wait only for the ids (not for seq_len): a page past the
  // request's length is masked, and a bad id flagged, when it is scored
  auto load_round = [&](int base) {
#pragma unroll
    for (int it = 0; it < kScoreIters; ++it) ids[it] = __shfl_sync(0xffffffffu, id_lane, it, L);
#pragma unroll
    for (int it = 0; it < kScoreIters; ++it) {
      const int pg = base + it * groups + grp;
      const int id = ids[it];
      live[it] = pg < p1 && id >= 0 && id < p.Lp;
      if (live[it]) {
        const int4* row = reinterpret_cast<const int4*>(slab_l + (size_t)id * HD);
#pragma unroll
        for (int c = 0; c < CPL; ++c) v[it][c] = __ldg(row + sub + c * L);
      }
    }
  };
  load_ids(p0);
  load_round(p0);

  // 2. q -> int8 with one symmetric scale per request (all heads), staged in
  //    shared memory; then the G query heads of each KV head summed
  //    (|sum| <= 127 * G fits int16)
  auto lane8 = [](const uint4& u, int i) -> float {
    const uint32_t w = i < 2 ? u.x : (i < 4 ? u.y : (i < 6 ? u.z : u.w));
    return __uint_as_float((i & 1 ? (w >> 16) : (w & 0xFFFFu)) << 16);
  };
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < kQV; ++j)
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(lane8(qraw[j], i)));
  amax = block_max(amax, red);
  const float s = amax / 127.0f;
#pragma unroll
  for (int j = 0; j < kQV; ++j) {
    const int vi = threadIdx.x + j * blockDim.x;
    if (vi >= nq16) continue;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int c = 0;
      if (amax > 0.0f) c = (int)fminf(fmaxf(rintf(lane8(qraw[j], i) / s), -127.0f), 127.0f);
      q8s[vi * 8 + i] = (int8_t)c;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < HD; e += blockDim.x) {
    const int h = e / p.D, d = e - h * p.D;
    int acc = 0;
    for (int g = 0; g < p.G; ++g) acc += q8s[(h * p.G + g) * p.D + d];
    qg[e] = (int16_t)acc;
  }
  __syncthreads();
  int qa[CPL][8];                  // this lane's q pairs
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const int* q2 = reinterpret_cast<const int*>(qg + (sub + c * L) * 16);
#pragma unroll
    for (int i = 0; i < 8; ++i) qa[c][i] = q2[i];
  }

  // 3. exact int32 dot products, reduced over the lanes of each page; the
  //    CTA walks its pages in rounds of kScoreIters groups.  The round's 8
  //    page sums are reduced over the L lanes together: at each of the first
  //    three levels a lane keeps half of its sums and trades the other half
  //    with its partner (8 -> 4 -> 2 -> 1 sums per lane, 7 shuffles), then a
  //    plain butterfly finishes the last log2(L) - 3 levels; lane sub ends up
  //    with page 4*b1 + 2*b2 + b3 of the round (b1, b2, b3: its lane bits L/2,
  //    L/4, L/8).  Integer sums: the order does not change the result.
  static_assert(kScoreIters == 8, "the transposed reduction halves 8 sums three times");
  const bool b1 = sub & (L >> 1), b2 = sub & (L >> 2), b3 = sub & (L >> 3);
  const int mine = (b1 ? 4 : 0) + (b2 ? 2 : 0) + (b3 ? 1 : 0);
  const bool writer = (sub & ((L >> 3) - 1)) == 0;
  for (int base = p0;;) {
    unsigned used = 0;
    if (base + groups * kScoreIters < p1) load_ids(base + groups * kScoreIters);
    auto dot = [&](int it) -> int {          // this lane's part of page it's score
      const int pg = base + it * groups + grp;
      const bool in = pg < p1 && pg < n_b;
      if (in && !live[it] && sub == 0) set_status(p.status, SSA_ST_BAD_ID);
      const bool use = in && live[it];
      used |= use ? 1u << it : 0u;
      int acc = 0;
      if (use) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const int w[4] = {v[it][c].x, v[it][c].y, v[it][c].z, v[it][c].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc = __dp2a_lo(qa[c][2 * j], w[j], acc);
            acc = __dp2a_hi(qa[c][2 * j + 1], w[j], acc);
          }
        }
      }
      return acc;
    };
    // pages i and i + 4 are scored together and traded at once, so that at
    // most two unreduced sums are live besides the four kept ones
    int a4[4], a2[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int lo = dot(i), hi = dot(i + 4);
      a4[i] = (b1 ? hi : lo) + __shfl_xor_sync(0xffffffffu, b1 ? lo : hi, L >> 1);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i)
      a2[i] = (b2 ? a4[i + 2] : a4[i]) +
              __shfl_xor_sync(0xffffffffu, b2 ? a4[i] : a4[i + 2], L >> 2);
    int a1 = (b3 ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, b3 ? a2[0] : a2[1], L >> 3);
    for (int o = L >> 4; o; o >>= 1) a1 += __shfl_xor_sync(0xffffffffu, a1, o);
    const int pg = base + mine * groups + grp;
    if (writer && pg < p1) out[pg] = (used >> mine) & 1u ? a1 : INT_MIN;
    base += groups * kScoreIters;
    if (base >= p1) break;
    load_round(base);
  }
}

// Shared memory of the score phase: qg [Hkv*D] int16, then q8s [Hq*D] int8.
__host__ __device__ inline int qg_bytes(int HD) { return (HD * 2 + 15) / 16 * 16; }
__host__ __device__ inline int q8_bytes(int HqD) { return (HqD + 15) / 16 * 16; }

template <int CPL>
__global__ void __launch_bounds__(kScoreThreads, CPL == 1 ? 3 : 2) index_score_kernel(ScoreParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  int16_t* qg = reinterpret_cast<int16_t*>(smem_raw);
  int8_t* q8s = reinterpret_cast<int8_t*>(smem_raw + qg_bytes(p.Hkv * p.D));
  __shared__ float red[33];
  pdl_wait();
  score_chunk<CPL>(p, qg, q8s, red);
}

// ---------------------------------------------------------------------------
// top-k select: one CTA per (layer, request)
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 1024;
constexpr int kSelCand = 64;       // a bin this small is ranked directly
// Upper bound on the static shared memory of the select (and fused index)
// kernels: histogram, scan scratch, a few scalars.
constexpr size_t kSelectStaticSmem = 2048;

struct SelectParams {
  const int32_t* scores;   // [n_layers][B][nmax]
  const int32_t* seq_lens;
  int32_t* sel;            // [n_layers][B][W]
  int32_t* n_sel;          // [n_layers][B]
  int32_t* status;
  int B, nmax, P, k, W;
};

// Top-k selection of one (layer, request) row of scores by the whole CTA.
// CG: the row was written by other CTAs of this kernel (read past L1).
template <bool CG>
__device__ void select_row(const int32_t* row, int n, int k, int W, int32_t* out,
                           int32_t* n_sel_out, int32_t* status, uint32_t* key) {
  __shared__ int hist[256];
  __shared__ int tmp[33];
  __shared__ uint32_t s_lo, s_hi, s_base;
  __shared__ int s_remaining, s_shift, s_bincnt, s_ncand;
  __shared__ uint32_t cbin[kSelCand];
  const int tid = threadIdx.x, nt = blockDim.x;
  const bool take_all = (n - 1 <= k);
  const int cand = n - 1;                // pages that compete; n-1 is forced
  uint32_t T = 0;
  int need_eq = 0;
  if (!take_all) {
    // order-preserving keys and their range
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    for (int i = tid; i < cand; i += nt) {
      const uint32_t kk = (uint32_t)(CG ? __ldcg(row + i) : row[i]) ^ 0x80000000u;
      key[i] = kk;
      lo = min(lo, kk);
      hi = max(hi, kk);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (tid == 0) { s_lo = 0xFFFFFFFFu; s_hi = 0u; s_remaining = k; }
    __syncthreads();
    if ((tid & 31) == 0) { atomicMin(&s_lo, lo); atomicMax(&s_hi, hi); }
    __syncthreads();
    // MSB-first radix search for the k-th largest key, restricted to the
    // keys' own range [lo, hi]: bins of 8 bits of (key - lo), starting at the
    // highest bit the range uses, so a narrow range needs fewer passes
    uint32_t base = s_lo;                 // keys below base are out
    const uint32_t range = s_hi - s_lo;
    int shift = range == 0 ? 0 : max(0, 32 - __clz((int)range) - 8);
    if (range >> 31) shift = 24;
    uint32_t span_hi = s_hi;              // candidates lie in [base, span_hi]
    for (;;) {
      for (int i = tid; i < 256; i += nt) hist[i] = 0;
      __syncthreads();
      for (int i = tid; i < cand; i += nt) {
        const uint32_t kk = key[i];
        if (kk >= base && kk <= span_hi) atomicAdd(&hist[((kk - base) >> shift) & 255], 1);
      }
      __syncthreads();
      if (tid < 32) {
        // lane l covers bins 255-8l down to 248-8l (largest first)
        int cnt[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) { cnt[j] = hist[255 - 8 * tid - j]; sum += cnt[j]; }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (tid >= o) incl += y;
        }
        const int rem = s_remaining;
        const unsigned hitm = __ballot_sync(0xffffffffu, incl >= rem);
        const int lane = __ffs(hitm) - 1;       // hitm != 0: rem <= candidates
        if (tid == lane) {
          int above = incl - sum;
          for (int j = 0; j < 8; ++j) {
            if (above + cnt[j] >= rem) {
              const uint32_t bin = (uint32_t)(255 - 8 * tid - j);
              s_remaining = rem - above;
              s_base = base + (bin << shift);
              s_shift = shift;
              s_bincnt = cnt[j];
              break;
            }
            above += cnt[j];
          }
        }
      }
      __syncthreads();
      base = s_base;
      if (shift == 0) break;
      span_hi = (uint32_t)min((unsigned long long)base + ((1ull << shift) - 1ull),
                              0xFFFFFFFFull);
      if (s_bincnt <= kSelCand) {
        // few keys left in the bin that holds the k-th largest: rank them
        // directly (each against all) instead of further radix passes
        if (tid == 0) s_ncand = 0;
        __syncthreads();
        for (int i = tid; i < cand; i += nt) {
          const uint32_t kk = key[i];
          if (kk >= base && kk <= span_hi) cbin[atomicAdd(&s_ncand, 1)] = kk;
        }
        __syncthreads();
        const int c = s_ncand, rem = s_remaining;
        for (int t = tid; t < c; t += nt) {
          const uint32_t x = cbin[t];
          int gt = 0, eq = 0;
          for (int j = 0; j < c; ++j) {
            gt += cbin[j] > x;
            eq += cbin[j] == x;
          }
          if (gt < rem && rem <= gt + eq) {   // x is the rem-th largest of the bin
            s_base = x;
            s_remaining = rem - gt;
          }
        }
        __syncthreads();
        base = s_base;
        break;
      }
      shift = shift >= 8 ? shift - 8 : 0;
    }
    T = base;                             // the k-th largest key
    need_eq = s_remaining;                // how many keys equal to T to take
  }

  // Ordered compaction, one packed scan.  Each page is "above" (forced, or
  // key > T: always taken), "equal" (key == T: the first need_eq in page
  // order are taken) or out.  A taken page's output slot is the number of
  // above pages before it plus min(equal pages before it, need_eq).
  const int per = (n + nt - 1) / nt;
  const int a0 = min(n, tid * per), a1 = min(n, a0 + per);
  auto kind = [&](int i) -> int {          // 2 above, 1 equal, 0 out
    if (take_all || i == cand) return 2;
    const uint32_t kk = key[i];
    return kk > T ? 2 : (kk == T ? 1 : 0);
  };
  int gt = 0, eq = 0;
  for (int i = a0; i < a1; ++i) {
    const int t = kind(i);
    gt += t == 2;
    eq += t == 1;
  }
  int packed_total;
  const int packed = block_exclusive_scan((gt << 16) | eq, tmp, packed_total);
  int g_before = packed >> 16, e_before = packed & 0xFFFF;
  const int total = (packed_total >> 16) + min(packed_total & 0xFFFF, need_eq);
  for (int i = a0; i < a1; ++i) {
    const int t = kind(i);
    if (t == 2) {
      const int off = g_before + min(e_before, need_eq);
      if (off < W) out[off] = i;
      ++g_before;
    } else if (t == 1) {
      if (e_before < need_eq) {
        const int off = g_before + e_before;
        if (off < W) out[off] = i;
      }
      ++e_before;
    }
  }
  const int kept = min(total, W);
  for (int i = kept + tid; i < W; i += nt) out[i] = -1;
  if (tid == 0) {
    *n_sel_out = kept;
    if (total > W) set_status(status, SSA_ST_DROP);
  }
}

__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(SelectParams p) {
  extern __shared__ uint32_t key[];      // [nmax] order-preserving score keys
  pdl_wait();
  const int b = blockIdx.x, li = blockIdx.y;
  const int n = min(p.nmax, (p.seq_lens[b] + p.P - 1) / p.P);
  select_row<false>(p.scores + ((size_t)li * p.B + b) * p.nmax, n, p.k, p.W,
                    p.sel + ((size_t)li * p.B + b) * p.W, p.n_sel + (size_t)li * p.B + b,
                    p.status, key);
}

// a1 + a2 in one launch: every CTA scores its chunk of pages; the last CTA of
// each (layer, request) to finish -- an atomic ticket, no CTA waits for
// another -- selects over the whole row.
struct FusedParams {
  ScoreParams s;
  int32_t* sel;          // [n_layers][B][W]
  int32_t* n_sel;        // [n_layers][B]
  int32_t* tickets;      // [n_layers][B], zero between calls
  int k, W, qg_bytes;
};

template <int CPL>
__global__ void __launch_bounds__(kScoreThreads, CPL == 1 ? 3 : 2) index_topk_kernel(FusedParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  int16_t* qg = reinterpret_cast<int16_t*>(smem_raw);
  int8_t* q8s = reinterpret_cast<int8_t*>(smem_raw + qg_bytes(p.s.Hkv * p.s.D));
  uint32_t* key = reinterpret_cast<uint32_t*>(smem_raw + p.qg_bytes);   // [nmax]
  __shared__ float red[33];
  __shared__ int s_last;
  pdl_trigger();
  pdl_wait();
  score_chunk<CPL>(p.s, qg, q8s, red);
  const int b = blockIdx.y, li = blockIdx.z;
  const size_t rb = (size_t)li * p.s.B + b;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&p.tickets[rb], 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int n = min(p.s.nmax, (p.s.seq_lens[b] + p.s.P - 1) / p.s.P);
  select_row<true>(p.s.scores + rb * p.s.nmax, n, p.k, p.W, p.sel + rb * p.W, p.n_sel + rb,
                   p.s.status, key);
  if (threadIdx.x == 0) p.tickets[rb] = 0;      // ready for the next call
}

// Pages per score CTA: the smallest multiple of one round (kScoreIters page
// groups) that keeps the grid within one wave of resident CTAs (occ per SM),
// so no CTA waits for a second wave.
int score_pages_per_cta(const Dims& d, int n_layers, int lanes, int occ) {
  const int round = kScoreIters * (kScoreThreads / lanes);
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 152;
  if (occ < 1) occ = 1;
  const long long rows = (long long)d.B * n_layers;
  long long chunks = (long long)sms * occ / rows;
  if (chunks < 1) chunks = 1;
  long long per = (d.nmax + chunks - 1) / chunks;
  per = (per + round - 1) / round * round;
  return (int)per;
}

}  // namespace

cudaError_t launch_index_scores(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                                const void* q, const int32_t* bt, const int32_t* seq_lens,
                                int32_t* scores, int32_t* status, cudaStream_t s) {
  ScoreParams p{};
  p.slab = c.slab;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.bt = bt;
  p.seq_lens = seq_lens;
  p.scores = scores;
  p.status = status;
  p.layer0 = layer0;
  p.Lp = d.Lp; p.B = d.B; p.Hq = d.Hq; p.Hkv = d.Hkv; p.G = d.G; p.D = d.D; p.P = d.P;
  p.nmax = d.nmax;
  const int chunks16 = d.Hkv * d.D / 16;       // 16-byte chunks per page row
  const int cpl = chunks16 > 32 ? 2 : 1;
  p.lanes = chunks16 / cpl;
  const size_t smem = (size_t)qg_bytes(d.Hkv * d.D) + q8_bytes(d.Hq * d.D);
  int occ = 1;
  cudaError_t oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &occ, cpl == 1 ? index_score_kernel<1> : index_score_kernel<2>, kScoreThreads, smem);
  if (oe != cudaSuccess) return oe;
  p.pages_per_cta = score_pages_per_cta(d, n_layers, p.lanes, occ);
  dim3 grid((d.nmax + p.pages_per_cta - 1) / p.pages_per_cta, d.B, n_layers);
  cudaError_t e = cpl == 1 ? launch_pdl(index_score_kernel<1>, grid, dim3(kScoreThreads), smem, s, p)
                           : launch_pdl(index_score_kernel<2>, grid, dim3(kScoreThreads), smem, s, p);
  count_launch();
  return e;
}

cudaError_t launch_index_topk(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                              const void* q, const int32_t* bt, const int32_t* seq_lens,
                              int32_t* scores, int32_t* sel, int32_t* n_sel, int32_t* tickets,
                              int32_t* status, cudaStream_t s) {
  FusedParams f{};
  ScoreParams& p = f.s;
  p.slab = c.slab;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.bt = bt;
  p.seq_lens = seq_lens;
  p.scores = scores;
  p.status = status;
  p.layer0 = layer0;
  p.Lp = d.Lp; p.B = d.B; p.Hq = d.Hq; p.Hkv = d.Hkv; p.G = d.G; p.D = d.D; p.P = d.P;
  p.nmax = d.nmax;
  const int chunks16 = d.Hkv * d.D / 16;
  const int cpl = chunks16 > 32 ? 2 : 1;
  p.lanes = chunks16 / cpl;
  f.sel = sel;
  f.n_sel = n_sel;
  f.tickets = tickets;
  f.k = d.k;
  f.W = d.W;
  f.qg_bytes = qg_bytes(d.Hkv * d.D) + q8_bytes(d.Hq * d.D);     // key[] after qg, q8s
  const size_t smem = (size_t)f.qg_bytes + (size_t)d.nmax * sizeof(uint32_t);
  int occ = 1;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &occ, cpl == 1 ? index_topk_kernel<1> : index_topk_kernel<2>, kScoreThreads, smem);
  if (e != cudaSuccess) return e;
  p.pages_per_cta = score_pages_per_cta(d, n_layers, p.lanes, occ);
  dim3 grid((d.nmax + p.pages_per_cta - 1) / p.pages_per_cta, d.B, n_layers);
  if (cpl == 1) {
    if (smem + kSelectStaticSmem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(index_topk_kernel<1>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
      return e;
    e = launch_pdl(index_topk_kernel<1>, grid, dim3(kScoreThreads), smem, s, f);
  } else {
    if (smem + kSelectStaticSmem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(index_topk_kernel<2>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)))
      return e;
    e = launch_pdl(index_topk_kernel<2>, grid, dim3(kScoreThreads), smem, s, f);
  }
  count_launch();
  return e;
}

cudaError_t launch_topk_select(const Dims& d, int n_layers, const int32_t* scores,
                               const int32_t* seq_lens, int32_t* sel, int32_t* n_sel,
                               int32_t* status, cudaStream_t s) {
  SelectParams p{scores, seq_lens, sel, n_sel, status, d.B, d.nmax, d.P, d.k, d.W};
  const size_t smem = (size_t)d.nmax * sizeof(uint32_t);
  if (smem + kSelectStaticSmem > 48 * 1024) {   // the default limit counts static memory too
    cudaError_t e = cudaFuncSetAttribute(topk_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_pdl(topk_select_kernel, dim3(d.B, n_layers), dim3(kSelThreads), smem, s, p);
  count_launch();
  return e;
}

}  // namespace ssa
