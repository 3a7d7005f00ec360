// ensure.cu -- a3 LRU ensure, a4 miss fetch, a5 block-table remap.
//
// FreeToken PR #499, "What" and "Design": the GPU's slots cache logical
// pages whose full copy lives in pinned host memory; the least recently used
// slot is reused first.  The update has fixed shapes and no host round trip,
// so a step can be captured in a CUDA graph; since the host copy is always
// current, evicting a page only rebinds its slot; each miss's K and V are
// then copied host -> device.  FreeToken PR #525: the copy includes the
// per-token fp8 scales, and the pool is sized so that a batch's whole
// selection fits.
//
// Order of events per layer (the pages state none; this is the reading the
// library takes, identical in the oracle):
//   1. U = distinct selected logical ids, ascending (a bitmap over the
//      logical ids and a popcount scan; a bitonic sort + dedup when the
//      bitmap does not fit the shared memory at hand);
//   2. hits: last_use = clock;
//   3. misses, ascending, take victims in order: free slots by slot id, then
//      bound slots not touched this step by (last_use, slot) -- the m
//      smallest keys found by an MSB radix select, then sorted;
//   4. rebind; 5. clock += 1.
// One CTA per layer: the state update is latency-bound (a few thousand keys),
// the copy that follows is a separate, wide kernel.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace ssa {
namespace {

constexpr int kEnsureThreads = 1024;

template <typename T>
__device__ void bitonic_sort_smem(T* a, int n /* power of two */) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool up = (i & k) == 0;
          const T x = a[i], y = a[ixj];
          if ((x > y) == up) { a[i] = y; a[ixj] = x; }
        }
      }
      __syncthreads();
    }
  }
}

struct EnsureParams {
  int32_t *slot_of, *page_of, *last_use, *clock;
  const int32_t* sel;    // [n_layers][B][W] page indices (W: the entries per request)
  const int32_t* bt;     // [B][nmax]
  int32_t* miss_page;    // [n_layers][mstride]
  int32_t* miss_slot;
  int32_t* n_miss;       // [n_layers]
  int32_t* phys;         // [n_layers][B][W] or null: the remapped table (a5 fused)
  int defer;             // misses are not copied here; phys marks them -2 - slot
  int32_t* status;
  int layer0, Lp, S, B, W, nmax, N2, mstride;
  // layers whose selections one state serves: 1 (one CTA per layer), or the
  // call's layer count (one CTA; the first layer's state, shared residency)
  int nsel;
  int has_mirror;
  // 0: the step's ensure (epoch = clock; hits touched; every miss bound; clock
  // advances).  1: a preload after the step's ensure (epoch = clock - 1;
  // slots of that epoch are never victims; misses beyond the victims left
  // are not fetched; the clock stays).
  int preload;
};

// Order-preserving victim key of slot s: 0xFFFFFFFF for a slot of the
// current epoch (never a victim), free slots first, then by last_use.
__device__ __forceinline__ uint32_t victim_key(const int32_t* page_of, const int32_t* last_use,
                                               int s, int32_t epoch) {
  const int32_t po = page_of[s], lu = last_use[s];
  if (po >= 0 && lu == epoch) return 0xFFFFFFFFu;             // touched this epoch
  const int32_t k = po < 0 ? -2 : lu;                          // free slots first
  return (uint32_t)k ^ 0x80000000u;
}

// Up to this many slots, the victim keys are read from global memory once and
// kept in shared memory; beyond it every radix pass reads them again.
constexpr int kSmemKeys = 16384;
// Up to this many misses, the victim order is found by all-pairs ranking
// (one pass, one barrier); beyond it by a bitonic sort.
constexpr int kRankMax = 1024;
// Upper bound on the ensure kernel's static shared memory (hist, scan
// scratch, a few scalars), budgeted beside its dynamic buffers.
constexpr size_t kEnsureStaticSmem = 2048;

template <bool KEYS_IN_SMEM>
__global__ void __launch_bounds__(kEnsureThreads) ensure_state_kernel(EnsureParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int N2 = p.N2;
  uint64_t* vic = reinterpret_cast<uint64_t*>(smem_raw);                   // [N2]
  uint32_t* ids = reinterpret_cast<uint32_t*>(smem_raw + (size_t)N2 * 8);   // [N2]
  uint32_t* keys = ids + N2;                                                 // [S] (KEYS_IN_SMEM)
  __shared__ int hist[256];
  __shared__ int tmp[33];
  __shared__ uint32_t s_prefix, s_lo, s_hi;
  __shared__ int s_remaining, s_nv, s_ncand;
  pdl_trigger();
  pdl_wait();

  const int li = blockIdx.x, layer = p.layer0 + li;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int BW = p.B * p.W * p.nsel;        // selection entries this state serves
  int32_t* slot_of = p.slot_of + (size_t)layer * p.Lp;
  int32_t* page_of = p.page_of + (size_t)layer * p.S;
  int32_t* last_use = p.last_use + (size_t)layer * p.S;
  int32_t* mpage = p.miss_page + (size_t)li * p.mstride;
  int32_t* mslot = p.miss_slot + (size_t)li * p.mstride;
  // the epoch whose slots are never victims, and the last_use given to the
  // ids this call touches or binds
  const int32_t clock = p.clock[layer] - (p.preload ? 1 : 0);

  // 0. every selected page already bound (the usual case of a resident pool):
  //    steps 1-4 reduce to touching the hits, and a touch is the same write
  //    whichever duplicate makes it, so one pass over the entries touches,
  //    translates (a5 fused) and looks for a miss or a bad id.  Only if it
  //    finds one does the full update below run; it makes the same touches
  //    and rewrites the whole table, so nothing of this pass is lost.
  {
    int32_t* phys0 = p.phys ? p.phys + (size_t)li * BW : nullptr;
    const int32_t* sel0 = p.sel + (size_t)li * BW;
    int odd = 0;
    for (int i = tid; i < BW; i += nt) {
      const int b = (i / p.W) % p.B;
      const int pg = sel0[i];
      int out = -1;
      if (pg >= 0) {
        const int id = pg < p.nmax ? p.bt[(size_t)b * p.nmax + pg] : -1;
        const int slot = id >= 0 && id < p.Lp ? slot_of[id] : -1;
        if (slot >= 0 && slot < p.S) {
          last_use[slot] = clock;
          out = slot;
        } else {
          odd = 1;
        }
      }
      if (phys0) phys0[i] = out;
    }
    if (!__syncthreads_or(odd)) {
      for (int i = tid; i < p.mstride; i += nt) { mpage[i] = -1; mslot[i] = -1; }
      if (tid == 0) {
        p.n_miss[li] = 0;
        if (!p.preload) p.clock[layer] = clock + 1;
      }
      return;
    }
  }

  // 1. the distinct selected logical ids, ascending, in ids[] (0xFFFFFFFF
  //    after them)
  auto selected_id = [&](int i) -> uint32_t {        // entry i of the batch's selection
    const int b = (i / p.W) % p.B;             // layer li + i / (B*W) in shared residency
    const int pg = p.sel[(size_t)li * p.B * p.W + i];
    if (pg < 0) return 0xFFFFFFFFu;
    const int id = pg < p.nmax ? p.bt[(size_t)b * p.nmax + pg] : -1;
    if (id >= 0 && id < p.Lp) return (uint32_t)id;
    set_status(p.status, SSA_ST_BAD_ID);
    return 0xFFFFFFFFu;
  };
  const int nw = (p.Lp + 31) / 32;
  if (nw <= 2 * N2) {
    // a bitmap over the logical ids (in the victim buffer, free until step
    // 3): set a bit per selected id, then each thread emits the set bits of
    // its words at its place in the popcount scan -- five barriers where a
    // sort of N2 keys takes log2(N2)^2/2
    uint32_t* bits = reinterpret_cast<uint32_t*>(vic);
    for (int w = tid; w < nw; w += nt) bits[w] = 0u;
    for (int i = tid; i < N2; i += nt) ids[i] = 0xFFFFFFFFu;
    __syncthreads();
    for (int i = tid; i < BW; i += nt) {
      const uint32_t id = selected_id(i);
      if (id != 0xFFFFFFFFu) atomicOr(&bits[id >> 5], 1u << (id & 31));
    }
    __syncthreads();
    const int wper = (nw + nt - 1) / nt;
    const int w0 = min(nw, tid * wper), w1 = min(nw, w0 + wper);
    int cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(bits[w]);
    int nd;
    int at = block_exclusive_scan(cnt, tmp, nd);
    for (int w = w0; w < w1; ++w) {
      uint32_t x = bits[w];
      while (x) {
        const int bit = __ffs(x) - 1;
        ids[at++] = (uint32_t)(w * 32 + bit);
        x &= x - 1u;
      }
    }
    __syncthreads();
  } else {
    for (int i = tid; i < N2; i += nt) ids[i] = i < BW ? selected_id(i) : 0xFFFFFFFFu;
    __syncthreads();
    bitonic_sort_smem(ids, N2);
  }

  // 2. hits are touched; misses ranked in ascending id order
  const int per = (N2 + nt - 1) / nt;
  const int a0 = min(N2, tid * per), a1 = min(N2, a0 + per);
  int my_miss = 0;
  for (int i = a0; i < a1; ++i) {
    const uint32_t id = ids[i];
    if (id == 0xFFFFFFFFu || (i > 0 && ids[i - 1] == id)) continue;
    const int slot = slot_of[id];
    if (slot >= p.S) { set_status(p.status, SSA_ST_BAD_ID); continue; }   // corrupt state
    if (slot >= 0) last_use[slot] = clock;
    else ++my_miss;
  }
  int m;
  int rank = block_exclusive_scan(my_miss, tmp, m);
  for (int i = a0; i < a1; ++i) {
    const uint32_t id = ids[i];
    if (id == 0xFFFFFFFFu || (i > 0 && ids[i - 1] == id)) continue;
    if (slot_of[id] < 0) mpage[rank++] = (int32_t)id;
  }
  __syncthreads();   // last_use touches and the miss list are visible block-wide

  if (m > 0) {
    // 3. the m smallest victim keys: MSB-first radix select on 32-bit keys
    if (KEYS_IN_SMEM) {
      for (int s = tid; s < p.S; s += nt) keys[s] = victim_key(page_of, last_use, s, clock);
    }
    auto key_of = [&](int s) -> uint32_t {
      return KEYS_IN_SMEM ? keys[s] : victim_key(page_of, last_use, s, clock);
    };
    // the candidates' key range (slots touched this step, key 0xFFFFFFFF,
    // are never victims): last_use values span a few hundred clocks, so
    // bins over the range need one or two passes where the full 32 bits
    // need four
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    int ncand = 0;
    for (int s = tid; s < p.S; s += nt) {
      const uint32_t kk = key_of(s);
      if (kk != 0xFFFFFFFFu) { lo = min(lo, kk); hi = max(hi, kk); ++ncand; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      ncand += __shfl_xor_sync(0xffffffffu, ncand, o);
    }
    if (tid == 0) { s_lo = 0xFFFFFFFFu; s_hi = 0u; s_nv = 0; s_ncand = 0; }
    __syncthreads();
    if ((tid & 31) == 0) { atomicMin(&s_lo, lo); atomicMax(&s_hi, hi); atomicAdd(&s_ncand, ncand); }
    __syncthreads();
    // a preload fetches the first misses (ascending id) that find a victim;
    // the ensure's capacity rule leaves it a victim for every miss
    if (s_ncand < m) {
      for (int i = s_ncand + tid; i < m; i += nt) mpage[i] = -1;
      m = s_ncand;
    }
    if (tid == 0) s_remaining = m;
    __syncthreads();
    if (m > 0) {
      // LSB-side radix search for the m-th smallest key within [base, span_hi]:
      // bins of 8 bits of (key - base), from the highest bit the range uses
      uint32_t base = s_lo, span_hi = s_hi;
      const uint32_t range = s_hi - s_lo;
      int shift = range == 0 ? 0 : max(0, 32 - __clz((int)range) - 8);
      if (range >> 31) shift = 24;
      for (;;) {
        for (int i = tid; i < 256; i += nt) hist[i] = 0;
        __syncthreads();
        for (int b0 = 0; b0 < p.S; b0 += nt) {        // uniform trip count
          const int s = b0 + tid;
          const uint32_t kk = s < p.S ? key_of(s) : 0xFFFFFFFFu;
          const bool use = s < p.S && kk >= base && kk <= span_hi && kk != 0xFFFFFFFFu;
          // one atomic per distinct bin per warp: last_use values cluster
          const int key = use ? (int)(((kk - base) >> shift) & 255) : -1 - (tid & 31);
          const unsigned peers = __match_any_sync(0xffffffffu, key);
          if (use && (tid & 31) == __ffs(peers) - 1) atomicAdd(&hist[key], __popc(peers));
        }
        __syncthreads();
        if (tid < 32) {
          int cnt[8], sum = 0;
  #pragma unroll
          for (int j = 0; j < 8; ++j) { cnt[j] = hist[8 * tid + j]; sum += cnt[j]; }
          int incl = sum;
  #pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (tid >= o) incl += y;
          }
          const int rem = s_remaining;
          const unsigned hit = __ballot_sync(0xffffffffu, incl >= rem);
          const int lane = __ffs(hit) - 1;
          if (tid == lane) {
            int below = incl - sum;
            for (int j = 0; j < 8; ++j) {
              if (below + cnt[j] >= rem) {
                s_remaining = rem - below;
                s_prefix = base + ((uint32_t)(8 * tid + j) << shift);
                break;
              }
              below += cnt[j];
            }
          }
        }
        __syncthreads();
        base = s_prefix;
        if (shift == 0) break;
        span_hi = (uint32_t)min((unsigned long long)base + ((1ull << shift) - 1ull), 0xFFFFFFFEull);
        shift = shift >= 8 ? shift - 8 : 0;
      }
      const uint32_t T = s_prefix;
      const int need_eq = s_remaining;
      // gather: keys below T (any order), then the need_eq lowest slots equal to T
      const int sper = (p.S + nt - 1) / nt;
      const int s0 = min(p.S, tid * sper), s1 = min(p.S, s0 + sper);
      int eq = 0;
      for (int s = s0; s < s1; ++s) {
        const uint32_t kk = key_of(s);
        if (kk < T) vic[atomicAdd(&s_nv, 1)] = ((uint64_t)kk << 32) | (uint32_t)s;
        else if (kk == T) ++eq;
      }
      int eqtot;
      int er = block_exclusive_scan(eq, tmp, eqtot);
      const int n_lt = m - need_eq;
      for (int s = s0; s < s1 && er < need_eq; ++s) {
        const uint32_t kk = key_of(s);
        if (kk == T) {
          if (er < need_eq) vic[n_lt + er] = ((uint64_t)kk << 32) | (uint32_t)s;
          ++er;
        }
      }
      __syncthreads();
      // 4. victim order: (key, slot) ascending.  The keys are distinct (slots
      //    are), so each victim's rank is the count of smaller keys.
      if (m <= kRankMax) {
        for (int i = tid; i < m; i += nt) {
          const uint64_t x = vic[i];
          int r = 0;
          for (int j = 0; j < m; ++j) r += vic[j] < x;
          ids[r] = (uint32_t)(x & 0xFFFFFFFFu);      // ids are no longer needed
        }
      } else {
        int M2 = 1;
        while (M2 < m) M2 <<= 1;
        for (int i = m + tid; i < M2; i += nt) vic[i] = ~0ull;
        __syncthreads();
        bitonic_sort_smem(vic, M2);
        for (int i = tid; i < m; i += nt) ids[i] = (uint32_t)(vic[i] & 0xFFFFFFFFu);
      }
      __syncthreads();

      // 5. rebind: i-th miss takes the i-th victim
      for (int i = tid; i < m; i += nt) {
        const int pg = mpage[i];
        const int v = (int)ids[i];
        const int old = page_of[v];
        if (old >= 0 && old < p.Lp) slot_of[old] = -1;
        slot_of[pg] = v;
        page_of[v] = pg;
        last_use[v] = clock;
        mslot[i] = v;
      }
    }
    if (tid == 0 && m > 0 && !p.has_mirror) set_status(p.status, SSA_ST_MISS_NO_MIRROR);
  }
  for (int i = m + tid; i < p.mstride; i += nt) { mpage[i] = -1; mslot[i] = -1; }
  __syncthreads();
  if (tid == 0) {
    p.n_miss[li] = m;
    if (!p.preload) p.clock[layer] = clock + 1;
  }
  if (p.phys) {
    // a5 fused: every selected page of the layer now has its slot (the
    // rebind above is visible block-wide), so translate the table here.
    // With deferred fetches the pages bound by this call (the misses, ids
    // ascending in the miss list) are marked -2 - slot: their bytes are not
    // in the slot yet, the attention fetches them.
    uint32_t* mids = reinterpret_cast<uint32_t*>(vic);      // free after the rebind
    const int nm = p.defer ? m : 0;
    for (int i = tid; i < nm; i += nt) mids[i] = (uint32_t)mpage[i];
    if (p.defer) __syncthreads();
    int32_t* phys = p.phys + (size_t)li * BW;
    const int32_t* sel = p.sel + (size_t)li * BW;
    for (int i = tid; i < BW; i += nt) {
      const int b = (i / p.W) % p.B;
      const int pg = sel[i];
      int out = -1;
      if (pg >= 0) {
        const int id = pg < p.nmax ? p.bt[(size_t)b * p.nmax + pg] : -1;
        if (id >= 0 && id < p.Lp) out = slot_of[id];
        if (out < 0) set_status(p.status, SSA_ST_UNRESOLVED);
        if (out >= 0 && nm > 0) {             // binary search of id among the misses
          int lo = 0, hi = nm;
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (mids[mid] < (uint32_t)id) lo = mid + 1; else hi = mid;
          }
          if (lo < nm && mids[lo] == (uint32_t)id) out = -2 - out;
        }
      }
      phys[i] = out;
    }
  }
}

// ---------------------------------------------------------------------------
// a4: copy each miss's page (K, V, fp8 scales) mirror -> slot.  Fixed grid of
// B*W entries per layer; entries past the device-side miss count return.
// 16-byte loads from pinned host memory over UVA, several in flight per
// thread, 16-byte stores to HBM.
// ---------------------------------------------------------------------------
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int kCopyChunk = kCopyThreads * kCopyUnroll;   // 16-byte units per CTA

struct CopyParams {
  const uint8_t *k_mir, *v_mir;
  const float *ks_mir, *vs_mir;
  uint8_t *k_pool, *v_pool;
  float *k_scale, *v_scale;
  const int32_t *miss_page, *miss_slot, *n_miss;
  int layer0, Lp, S, BW, P, fp8;
  int shared;             // one miss list (the first layer's) for every layer
  long long page_bytes;   // one page, all KV heads
};

__global__ void __launch_bounds__(kCopyThreads) miss_copy_kernel(CopyParams p) {
  pdl_trigger();
  pdl_wait();
  const int entry = blockIdx.y, li = blockIdx.z, layer = p.layer0 + li;
  const int lst = p.shared ? 0 : li;          // the miss list this layer copies
  if (entry >= p.n_miss[lst] || p.k_mir == nullptr) return;
  const int pg = p.miss_page[(size_t)lst * p.BW + entry];
  const int slot = p.miss_slot[(size_t)lst * p.BW + entry];
  if (pg < 0 || pg >= p.Lp || slot < 0 || slot >= p.S) return;
  const long long pb16 = p.page_bytes / 16;
  const long long sc16 = p.fp8 ? (long long)p.P * 4 / 16 : 0;
  const long long total = 2 * pb16 + 2 * sc16;
  const size_t mp = (size_t)layer * p.Lp + pg, ps = (size_t)layer * p.S + slot;
  // 16-byte unit idx of the concatenation [K page | V page | K scales | V scales]
  auto locate = [&](long long idx, const uint4*& src, uint4*& dst) {
    if (idx < pb16) {
      src = reinterpret_cast<const uint4*>(p.k_mir + mp * p.page_bytes) + idx;
      dst = reinterpret_cast<uint4*>(p.k_pool + ps * p.page_bytes) + idx;
    } else if (idx < 2 * pb16) {
      idx -= pb16;
      src = reinterpret_cast<const uint4*>(p.v_mir + mp * p.page_bytes) + idx;
      dst = reinterpret_cast<uint4*>(p.v_pool + ps * p.page_bytes) + idx;
    } else if (idx < 2 * pb16 + sc16) {
      idx -= 2 * pb16;
      src = reinterpret_cast<const uint4*>(p.ks_mir + mp * p.P) + idx;
      dst = reinterpret_cast<uint4*>(p.k_scale + ps * p.P) + idx;
    } else {
      idx -= 2 * pb16 + sc16;
      src = reinterpret_cast<const uint4*>(p.vs_mir + mp * p.P) + idx;
      dst = reinterpret_cast<uint4*>(p.v_scale + ps * p.P) + idx;
    }
  };
  uint4 buf[kCopyUnroll];
  uint4* dst[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const long long idx = (long long)blockIdx.x * kCopyChunk + u * kCopyThreads + threadIdx.x;
    dst[u] = nullptr;
    if (idx < total) {
      const uint4* src;
      locate(idx, src, dst[u]);
      buf[u] = *src;
    }
  }
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u)
    if (dst[u]) *dst[u] = buf[u];
}

// ---------------------------------------------------------------------------
// a5: phys[b][i] = slot_of[bt[b][sel[b][i]]], -1 for padding.
// ---------------------------------------------------------------------------
__global__ void remap_kernel(const int32_t* slot_of, const int32_t* sel, const int32_t* bt,
                             int32_t* phys, int32_t* status, int layer0, int n_layers, int Lp,
                             int B, int W, int nmax) {
  pdl_trigger();
  pdl_wait();
  const long long n = (long long)n_layers * B * W;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int li = (int)(i / ((long long)B * W));
    const int b = (int)((i / W) % B);
    const int pg = sel[i];
    int out = -1;
    if (pg >= 0) {
      const int id = pg < nmax ? bt[(size_t)b * nmax + pg] : -1;
      if (id >= 0 && id < Lp) out = slot_of[(size_t)(layer0 + li) * Lp + id];
      else set_status(status, SSA_ST_BAD_ID);
      if (out < 0) set_status(status, SSA_ST_UNRESOLVED);
    }
    phys[i] = out;
  }
}

}  // namespace

int ensure_sort_width(const Dims& d, int nsel) {
  int n = 2;
  while (n < d.B * d.W * nsel) n <<= 1;
  return n;
}

namespace {

cudaError_t launch_state(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                         const int32_t* sel, int width, int preload, const int32_t* bt,
                         int32_t* miss_page, int32_t* miss_slot, int32_t* n_miss,
                         int32_t* phys, int32_t* status, cudaStream_t s, bool shared = false,
                         bool defer = false) {
  EnsureParams p{};
  p.phys = phys;
  p.defer = defer ? 1 : 0;
  p.nsel = shared ? n_layers : 1;
  p.slot_of = c.slot_of; p.page_of = c.page_of; p.last_use = c.last_use; p.clock = c.clock;
  p.sel = sel; p.bt = bt; p.miss_page = miss_page; p.miss_slot = miss_slot; p.n_miss = n_miss;
  p.status = status;
  p.layer0 = layer0; p.Lp = d.Lp; p.S = d.S; p.B = d.B; p.W = width; p.nmax = d.nmax;
  p.N2 = ensure_sort_width(d, p.nsel);
  p.mstride = d.B * d.W * p.nsel;
  p.preload = preload;
  p.has_mirror = c.k_mirror != nullptr;
  // small batches and pools: 256 threads (cheaper barriers); else 1024
  const int threads = (p.N2 <= 1024 && d.S <= 4096) ? 256 : kEnsureThreads;
  // the slots' victim keys stay in shared memory when they fit beside the id
  // and victim buffers (and the kernel's static shared memory) within the
  // device's per-CTA limit; otherwise every radix pass reads them again
  const size_t base = (size_t)p.N2 * 12;
  const size_t with_keys = base + (size_t)d.S * 4;
  const bool keys_in_smem =
      d.S <= kSmemKeys && with_keys + kEnsureStaticSmem <= (size_t)current_device_info().smem_optin;
  const size_t smem = keys_in_smem ? with_keys : base;
  auto k = keys_in_smem ? ensure_state_kernel<true> : ensure_state_kernel<false>;
  // the default limit (48 KiB) covers static and dynamic shared memory together
  if (smem + kEnsureStaticSmem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_pdl(k, dim3(shared ? 1 : n_layers), dim3(threads), smem, s, p);
  count_launch();
  return e;
}

}  // namespace

cudaError_t launch_ensure_state(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                                const int32_t* sel, const int32_t* bt, int32_t* miss_page,
                                int32_t* miss_slot, int32_t* n_miss, int32_t* phys,
                                int32_t* status, cudaStream_t s) {
  return launch_state(d, c, layer0, n_layers, sel, d.W, 0, bt, miss_page, miss_slot, n_miss,
                      phys, status, s);
}

cudaError_t launch_ensure_state_deferred(const Dims& d, const ssa_cache& c, int layer0,
                                         int n_layers, const int32_t* sel, const int32_t* bt,
                                         int32_t* miss_page, int32_t* miss_slot, int32_t* n_miss,
                                         int32_t* phys, int32_t* status, cudaStream_t s) {
  return launch_state(d, c, layer0, n_layers, sel, d.W, 0, bt, miss_page, miss_slot, n_miss,
                      phys, status, s, false, true);
}

cudaError_t launch_ensure_state_shared(const Dims& d, const ssa_cache& c, int layer0,
                                       int n_layers, const int32_t* sel, const int32_t* bt,
                                       int32_t* miss_page, int32_t* miss_slot, int32_t* n_miss,
                                       int32_t* phys, int32_t* status, cudaStream_t s) {
  return launch_state(d, c, layer0, n_layers, sel, d.W, 0, bt, miss_page, miss_slot, n_miss,
                      phys, status, s, true);
}

cudaError_t launch_preload_state(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                                 const int32_t* cand, int width, const int32_t* bt,
                                 int32_t* miss_page, int32_t* miss_slot, int32_t* n_miss,
                                 int32_t* status, cudaStream_t s) {
  return launch_state(d, c, layer0, n_layers, cand, width, 1, bt, miss_page, miss_slot, n_miss,
                      nullptr, status, s);
}

cudaError_t launch_miss_copy(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                             const int32_t* miss_page, const int32_t* miss_slot,
                             const int32_t* n_miss, int32_t* status, cudaStream_t s,
                             bool shared) {
  (void)status;
  if (c.k_mirror == nullptr) return cudaSuccess;   // nothing to fetch from (flagged by ensure)
  CopyParams p{};
  p.k_mir = static_cast<const uint8_t*>(c.k_mirror);
  p.v_mir = static_cast<const uint8_t*>(c.v_mirror);
  p.ks_mir = c.k_scale_mirror; p.vs_mir = c.v_scale_mirror;
  p.k_pool = static_cast<uint8_t*>(c.k_pool); p.v_pool = static_cast<uint8_t*>(c.v_pool);
  p.k_scale = c.k_scale; p.v_scale = c.v_scale;
  p.miss_page = miss_page; p.miss_slot = miss_slot; p.n_miss = n_miss;
  p.layer0 = layer0; p.Lp = d.Lp; p.S = d.S; p.P = d.P; p.fp8 = d.fp8;
  p.shared = shared ? 1 : 0;
  p.BW = d.B * d.W * (shared ? n_layers : 1);   // list stride and entries per list
  p.page_bytes = (long long)d.page_bytes();
  const long long total16 = 2 * p.page_bytes / 16 + (d.fp8 ? 2LL * d.P * 4 / 16 : 0);
  dim3 grid((unsigned)((total16 + kCopyChunk - 1) / kCopyChunk), p.BW, n_layers);
  cudaError_t e = launch_pdl(miss_copy_kernel, grid, dim3(kCopyThreads), 0, s, p);
  count_launch();
  return e;
}

cudaError_t launch_remap(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                         const int32_t* sel, const int32_t* bt, int32_t* phys,
                         int32_t* status, cudaStream_t s) {
  const long long n = (long long)n_layers * d.B * d.W;
  const int threads = 256;
  const int blocks = (int)((n + threads - 1) / threads);
  cudaError_t e = launch_pdl(remap_kernel, dim3(blocks), dim3(threads), 0, s,
                             (const int32_t*)c.slot_of, sel, bt, phys, status, layer0, n_layers,
                             d.Lp, d.B, d.W, d.nmax);
  count_launch();
  return e;
}

}  // namespace ssa
