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
constexpr int kScoreIters = 4;     // pages per lane group per CTA (loads in flight)

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

// CPL: 16-byte chunks per lane (HD = 16 * lanes * CPL).
template <int CPL>
__global__ void __launch_bounds__(kScoreThreads) index_score_kernel(ScoreParams p) {
  extern __shared__ int16_t qg[];  // [Hkv][D] group sums of q8
  __shared__ float red[33];
  pdl_wait();
  const int li = blockIdx.z, b = blockIdx.y;
  const int HD = p.Hkv * p.D;
  const int L = p.lanes;
  const int sub = threadIdx.x & (L - 1), grp = threadIdx.x / L;
  const int groups = blockDim.x / L;

  // 1. issue this thread's slab loads first: they do not depend on q, so the
  //    q quantisation below runs while they are in flight
  const int n_b = min(p.nmax, (p.seq_lens[b] + p.P - 1) / p.P);
  const int p0 = blockIdx.x * p.pages_per_cta;             // pages_per_cta = groups * iters
  const int8_t* slab_l = p.slab + (size_t)(p.layer0 + li) * p.Lp * HD;
  int4 v[kScoreIters][CPL];
  bool live[kScoreIters];
#pragma unroll
  for (int it = 0; it < kScoreIters; ++it) {
    const int pg = p0 + it * groups + grp;
    live[it] = false;
    if (pg < p.nmax && pg < n_b) {
      const int id = p.bt[(size_t)b * p.nmax + pg];
      if (id >= 0 && id < p.Lp) {
        live[it] = true;
        const int4* row = reinterpret_cast<const int4*>(slab_l + (size_t)id * HD);
#pragma unroll
        for (int c = 0; c < CPL; ++c) v[it][c] = __ldg(row + sub + c * L);
      } else if (sub == 0) {
        set_status(p.status, SSA_ST_BAD_ID);
      }
    }
  }

  // 2. q -> int8 with one symmetric scale per request (all heads), then the
  //    G query heads of each KV head summed: |sum| <= 127 * G fits int16
  const __nv_bfloat16* qb = p.q + ((size_t)li * p.B + b) * p.Hq * p.D;
  float amax = 0.0f;
  for (int i = threadIdx.x; i < p.Hq * p.D; i += blockDim.x)
    amax = fmaxf(amax, fabsf(__bfloat162float(qb[i])));
  amax = block_max(amax, red);
  const float s = amax / 127.0f;
  for (int e = threadIdx.x; e < HD; e += blockDim.x) {
    const int h = e / p.D, d = e - h * p.D;
    int acc = 0;
    for (int g = 0; g < p.G; ++g) {
      int c = 0;
      if (amax > 0.0f) {
        float r = rintf(__bfloat162float(qb[(h * p.G + g) * p.D + d]) / s);
        c = (int)fminf(fmaxf(r, -127.0f), 127.0f);
      }
      acc += c;
    }
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

  // 3. exact int32 dot products, reduced over the lanes of each page
  int32_t* out = p.scores + ((size_t)li * p.B + b) * p.nmax;
#pragma unroll
  for (int it = 0; it < kScoreIters; ++it) {
    const int pg = p0 + it * groups + grp;
    int acc = 0;
    if (live[it]) {
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
    for (int o = L >> 1; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (sub == 0 && pg < p.nmax) out[pg] = live[it] ? acc : INT_MIN;
  }
}

// Histogram increment with one atomic per distinct bin per warp (keys often
// share their top digits, which would serialise plain atomics).  Every lane
// of the warp must call it; lanes with use == false add nothing.
__device__ __forceinline__ void hist_add_warp(int* hist, bool use, int bin) {
  const int lane = threadIdx.x & 31;
  const int key = use ? bin : -1 - lane;
  const unsigned peers = __match_any_sync(0xffffffffu, key);
  if (use && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
}

// ---------------------------------------------------------------------------
// top-k select: one CTA per (layer, request)
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 1024;

struct SelectParams {
  const int32_t* scores;   // [n_layers][B][nmax]
  const int32_t* seq_lens;
  int32_t* sel;            // [n_layers][B][W]
  int32_t* n_sel;          // [n_layers][B]
  int32_t* status;
  int B, nmax, P, k, W;
};

__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(SelectParams p) {
  extern __shared__ uint32_t key[];      // [nmax] order-preserving score keys
  __shared__ int hist[256];
  __shared__ int tmp[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_remaining;
  pdl_wait();
  const int b = blockIdx.x, li = blockIdx.y;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int n = min(p.nmax, (p.seq_lens[b] + p.P - 1) / p.P);
  const int32_t* row = p.scores + ((size_t)li * p.B + b) * p.nmax;
  int32_t* out = p.sel + ((size_t)li * p.B + b) * p.W;

  const bool take_all = (n - 1 <= p.k);
  const int cand = n - 1;                // pages that compete; n-1 is forced
  uint32_t T = 0;
  int need_eq = 0;
  if (!take_all) {
    for (int i = tid; i < cand; i += nt) key[i] = (uint32_t)row[i] ^ 0x80000000u;
    if (tid == 0) { s_prefix = 0; s_remaining = p.k; }
    uint32_t mask = 0;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += nt) hist[i] = 0;
      __syncthreads();
      const uint32_t prefix = s_prefix;
      for (int base = 0; base < cand; base += nt) {       // uniform trip count
        const int i = base + tid;
        const uint32_t kk = i < cand ? key[i] : 0u;
        hist_add_warp(hist, i < cand && (kk & mask) == prefix, (int)((kk >> shift) & 255));
      }
      __syncthreads();
      if (tid < 32) {
        // lane l covers digits 255-8l down to 248-8l (largest first)
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
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= rem);
        const int lane = __ffs(hit) - 1;       // hit != 0: rem <= total
        if (tid == lane) {
          int above = incl - sum;
          for (int j = 0; j < 8; ++j) {
            if (above + cnt[j] >= rem) {
              s_remaining = rem - above;
              s_prefix = prefix | ((uint32_t)(255 - 8 * tid - j) << shift);
              break;
            }
            above += cnt[j];
          }
        }
      }
      mask |= 0xFFu << shift;
      __syncthreads();
    }
    T = s_prefix;
    need_eq = s_remaining;
  }

  // ranks in page order: contiguous runs of pages per thread
  const int per = (n + nt - 1) / nt;
  const int a0 = min(n, tid * per), a1 = min(n, a0 + per);
  int eq_before = 0;
  if (!take_all) {
    int eq = 0;
    for (int i = a0; i < a1; ++i) eq += (i < cand && key[i] == T);
    int tot;
    eq_before = block_exclusive_scan(eq, tmp, tot);
  }
  int mine = 0;
  {
    int e = eq_before;
    for (int i = a0; i < a1; ++i) {
      bool f;
      if (take_all || i == cand) f = true;
      else if (key[i] > T) f = true;
      else if (key[i] == T) f = (e++ < need_eq);
      else f = false;
      mine += f;
    }
  }
  int total;
  int off = block_exclusive_scan(mine, tmp, total);
  {
    int e = eq_before;
    for (int i = a0; i < a1; ++i) {
      bool f;
      if (take_all || i == cand) f = true;
      else if (key[i] > T) f = true;
      else if (key[i] == T) f = (e++ < need_eq);
      else f = false;
      if (f) {
        if (off < p.W) out[off] = i;
        ++off;
      }
    }
  }
  const int kept = min(total, p.W);
  for (int i = kept + tid; i < p.W; i += nt) out[i] = -1;
  if (tid == 0) {
    p.n_sel[(size_t)li * p.B + b] = kept;
    if (total > p.W) set_status(p.status, SSA_ST_DROP);
  }
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
  p.pages_per_cta = kScoreIters * (kScoreThreads / p.lanes);
  dim3 grid((d.nmax + p.pages_per_cta - 1) / p.pages_per_cta, d.B, n_layers);
  const size_t smem = (size_t)d.Hkv * d.D * sizeof(int16_t);
  cudaError_t e = cpl == 1 ? launch_pdl(index_score_kernel<1>, grid, dim3(kScoreThreads), smem, s, p)
                           : launch_pdl(index_score_kernel<2>, grid, dim3(kScoreThreads), smem, s, p);
  count_launch();
  return e;
}

cudaError_t launch_topk_select(const Dims& d, int n_layers, const int32_t* scores,
                               const int32_t* seq_lens, int32_t* sel, int32_t* n_sel,
                               int32_t* status, cudaStream_t s) {
  SelectParams p{scores, seq_lens, sel, n_sel, status, d.B, d.nmax, d.P, d.k, d.W};
  const size_t smem = (size_t)d.nmax * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(topk_select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_pdl(topk_select_kernel, dim3(d.B, n_layers), dim3(kSelThreads), smem, s, p);
  count_launch();
  return e;
}

}  // namespace ssa
