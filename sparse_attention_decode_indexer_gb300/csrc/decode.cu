// decode.cu -- a6 sparse paged GQA decode attention and a7 split merge.
//
// FreeToken PR #499, "Design": after ensure, the block table is translated
// logical -> physical and the sparse paged attention runs on it, reading only
// the selected pages.  For request b, KV head h and its G query heads:
//     o[g] = sum_t softmax_t(sm_scale * q[g] . K[t]) V[t]
// over the valid tokens of the selected pages (fp8: K = code * k_scale[t],
// V = code * v_scale[t]).
//
// Design (sm_103a):
//   * work partition: a "unit" is one (layer, request, KV head); each unit
//     weighs w = min(n_max, k + 1) tiles (the selection size of a request
//     with at least k + 1 pages).  The units' tiles form one line of
//     T = units * w tiles that a single wave of CTAs cuts into equal
//     contiguous ranges, so every SM streams the same number of pages
//     whatever the unit count.  A CTA's range holds whole units and at most
//     two pieces of units it shares with its neighbours; a piece maps its
//     share of the unit's weight onto the same share of the unit's valid
//     selected pages;
//   * one producer warp walks the range: per unit it reads the sel/phys row,
//     counts the valid entries and streams its piece's pages (one KV head,
//     P tokens of K and V) into shared memory with TMA tiled copies (128-byte
//     swizzle), plus the fp8 per-token scales with bulk copies, through an
//     mbarrier ring.  Each stage carries a small descriptor (first/last page
//     of a piece, valid tokens, unit); the first page of a piece also brings
//     the unit's G query rows.  Empty pieces and the end of the range travel
//     as stages without data;
//   * four consumer warps each take 16-token blocks: QK^T with the tokens as
//     the MMA rows (A = K, B = q^T, N = 8 query heads) and PV with d as the
//     rows (A = V^T, B = P^T, the probabilities transposed in registers by
//     movmatrix), fp32 accumulate, online softmax in the log2 domain against
//     a lazy reference (the running maximum moves only when a score exceeds
//     it by 2^8, so most blocks skip the cross-lane reductions);
//   * bf16 K/V: m16n8k16 bf16 MMAs, fragments by ldmatrix (V transposed by
//     ldmatrix.trans);
//   * fp8 K/V: QK as m16n8k32 e4m3 MMAs on the raw K codes against q scaled
//     by a power of two and split into two e4m3 terms (hi + lo); PV as
//     m16n8k16 f16 MMAs on the V codes converted exactly to f16; fragments
//     by ldmatrix.  The K scale multiplies the fp32 score, and the V scale
//     folds into the probabilities (relative to a running power-of-two
//     reference, so the f16 operand never overflows).  V is stored d-major
//     in the pool ([Hkv][D][P]) so that the 8-bit reads run along tokens, the
//     reduction axis of PV;
//   * at the end of a piece each consumer warp leaves its softmax state in
//     shared memory and streams on; a sixth warp combines the 4 states: a
//     whole unit becomes its output, a shared unit's piece an (m, l, o)
//     partial that it publishes (GPU-scope fence, atomic ticket); the last
//     piece of a unit to arrive merges the unit's partials into the output.
//     No CTA ever waits for another, no consumer warp for another;
//   * every stage's descriptor carries its index in the CTA's stream, which
//     the consumers check against the stage they waited for
//     (SSA_ST_INTERNAL if it ever differs);
//   * host-tail mode (ssa_sparse_paged_decode_host_tail): the producer
//     resolves each selected page through slot_of itself; a page without a
//     slot is copied from the pinned host mirror by the producer warp's
//     16-byte cp.async loads over UVA into the same swizzled stage layout,
//     the stage's barrier tracking those copies instead of a TMA byte count;
//   * fetch mode (ssa_sparse_paged_decode_fetch): entries the deferred
//     ensure marked -2 - slot are read from the mirror the same way, and the
//     consumer warps also write them into their slots;
//   * the merges of a unit's pieces (by the merge warp or by the consumer
//     warps) run the same online recurrence in piece order, so the output
//     does not depend on which piece finishes last.
// The work is HBM-bound (8 flop/byte bf16, 16 fp8): the tensor cores carry
// the G-row tiles, the memory system sets the pace where a launch is large
// enough; the fp8 consumers' issue and ALU work limit the rest.
#include <cudaTypedefs.h>
#include <cuda.h>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>

#include "common.cuh"
#include "internal.h"

namespace ssa {
namespace {

constexpr int kD = 128;
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kMergeWarp = kConsumerWarps + 1;
constexpr int kDecodeThreads = kConsumers + 64;
constexpr int kMaxG = 8;
constexpr int kWindow = 32;          // producer compaction window (entries)
constexpr int kMaxStages = 12;
constexpr float kSlack = 8.0f;     // log2 headroom of the running softmax reference
constexpr int kSmemPerSm = 228 * 1024;
constexpr int kSmemPerCtaMax = 227 * 1024;
constexpr int kSmemReservedPerCta = 1024;

// kernel modes
constexpr int kResident = 0;   // every selected page in its pool slot (phys)
constexpr int kHostTail = 1;   // slots from slot_of; pages without one read from the mirror
constexpr int kFetch = 2;      // phys marks pages bound but not copied (-2 - slot): read
                               // from the mirror, used, and written into their slots

// stage descriptor flags
constexpr int kFirst = 1;   // first page of a piece: the stage also holds q
constexpr int kLast = 2;    // last page of a piece: flush after it
constexpr int kEmpty = 4;   // a piece without pages (no data in the stage)
constexpr int kDone = 8;    // end of the CTA's range
constexpr int kFinal = 16;  // with kLast / kEmpty: the CTA's last piece
constexpr int kWriteBack = 32;  // fetch mode: the stage's page goes to its slot too

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

template <bool FP8, int P>
struct Cfg {
  static constexpr int kTileBytes = P * kD * (FP8 ? 1 : 2);      // one KV head of one page
  static constexpr int kScaleBytes = FP8 ? 2 * P * 4 : 0;
  static constexpr int kQOff = 2 * kTileBytes + kScaleBytes;
  static constexpr int kQBytes = kMaxG * kD * 2;
  static constexpr int kStageBytes = round_up(kQOff + kQBytes, 1024);
  static constexpr int kCombineBytes = kConsumerWarps * kMaxG * kD * 4 + 2 * kConsumerWarps * kMaxG * 4;
  // alignment slack, combine area, producer window, descriptors and barriers
  static constexpr int kFixed = 1024 + kCombineBytes + kWindow * 12 + kMaxStages * 36 + 64;
  // two CTAs per SM when at least two stages fit beside the second CTA
  static constexpr int kStages2 = (kSmemPerSm / 2 - kSmemReservedPerCta - kFixed) / kStageBytes;
  static constexpr int kCtasPerSm = kStages2 >= 2 ? 2 : 1;
  static constexpr int kStagesFit =
      kCtasPerSm == 2 ? kStages2 : (kSmemPerCtaMax - kFixed) / kStageBytes;
  static constexpr int kStages = kStagesFit > kMaxStages ? kMaxStages : kStagesFit;
  static constexpr int kBlocks = P / 16;                          // 16-token blocks per page
  // log2 of the fp8 V^T row swizzle span in 16-byte units (row = P bytes)
  static constexpr int kVSwz = P >= 128 ? 3 : (P == 64 ? 2 : (P == 32 ? 1 : 0));
  static_assert(kStages >= 2, "at least two stages");
  static_assert(kQOff % 16 == 0, "q rows need a 16-byte aligned bulk copy");
};

struct DecodeParams {
  const __nv_bfloat16* q;   // [n_layers][B][Hq][D]
  const int32_t* sel;       // [n_layers][B][W]
  const int32_t* phys;
  const int32_t* seq_lens;
  const float* k_scale;     // [Lyr][S][P]
  const float* v_scale;
  __nv_bfloat16* out;       // [n_layers][B][Hq][D]
  float* part_o;            // [n_ctas][2][G][D]
  float* part_ml;           // [n_ctas][2][G][2]
  int32_t* tickets;         // [units] piece counters, zero between calls
  int32_t* status;
  int T, tq, tr;             // tiles (units * w); CTA c holds [c*tq + min(c, tr), ...)
  int layer0, B, Hq, Hkv, G, W, S, w;
  float sm_log2;            // sm_scale * log2(e)
  // host-tail mode (phys unused): each selected page is resolved through
  // slot_of; pages without a slot are read from the pinned mirror over UVA
  int host_tail;
  int Lp, nmax;
  uint8_t *k_pool, *v_pool;       // fetch mode: where fetched pages are written back
  const int32_t* bt;        // [B][nmax]
  const int32_t* slot_of;   // [Lyr][Lp]
  const uint8_t *k_mir, *v_mir;   // [Lyr][Lp][page bytes]
  const float *ks_mir, *vs_mir;   // [Lyr][Lp][P]
};

// 16-byte asynchronous copy global (device or mapped host memory) -> shared
__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}

// The mbarrier tracks this thread's earlier cp.async copies: an arrival once
// they complete (the expected count is raised first, so the net change is
// zero and the phase waits for the copies).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// byte offset inside a tile whose rows were written by TMA with a
// 2^swz x 16-byte swizzle (bits [4, 4+swz) ^= bits [7, 7+swz))
__device__ __forceinline__ uint32_t swz(uint32_t a, int bits) {
  return a ^ (((a >> 7) & ((1u << bits) - 1u)) << 4);
}

// 1/x for x a positive normal power of two, exactly, without a division.
__device__ __forceinline__ float pow2_rcp(float x) {
  return __uint_as_float(0x7F000000u - __float_as_uint(x));
}

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

// |x| max of the 8 bf16 values in a 16-byte word
__device__ __forceinline__ float bf16x8_absmax(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, __uint_as_float((w[i] << 16) & 0x7FFF0000u));
    m = fmaxf(m, __uint_as_float(w[i] & 0x7FFF0000u));
  }
  return m;
}

// The merge of a unit's pieces (a7), written once so that the merge warp and
// the consumer warps, whichever holds the unit's last piece to finish, do
// the same arithmetic in the same order and the output does not depend on
// which piece arrives last: per (head, 4 columns) an online max / sum /
// weighted sum over the pieces in piece order.
__device__ __forceinline__ void merge_online(float& M, float& L, float4& acc, float2 ml,
                                             float4 x) {
  if (ml.x == -INFINITY) return;                // a piece with no token of this unit
  const float mn = fmaxf(M, ml.x);
  const float a = fast_exp2(M - mn), b = fast_exp2(ml.x - mn);
  L = fmaf(ml.y, b, L * a);
  acc.x = fmaf(x.x, b, acc.x * a);
  acc.y = fmaf(x.y, b, acc.y * a);
  acc.z = fmaf(x.z, b, acc.z * a);
  acc.w = fmaf(x.w, b, acc.w * a);
  M = mn;
}

// First tile of CTA c (the first tr CTAs hold tq + 1 tiles, the others
// tq), and the CTA that holds tile t (the inverse).
__device__ __forceinline__ int tile_begin(const DecodeParams& p, int c) {
  return c * p.tq + min(c, p.tr);
}
__device__ __forceinline__ int cta_of(const DecodeParams& p, int t) {
  const int big = p.tr * (p.tq + 1);
  return t < big ? t / (p.tq + 1) : p.tr + (t - big) / p.tq;
}

// MODE: kResident, kHostTail or kFetch -- separate instantiations, so that
// the resident path carries none of the other modes' code
template <bool FP8, int P, int MODE>
__global__ void __launch_bounds__(kDecodeThreads, Cfg<FP8, P>::kCtasPerSm)
decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV) {
  constexpr bool HT = MODE == kHostTail;
  constexpr bool FT = MODE == kFetch;
  constexpr bool WARP_ISSUE = HT || FT;     // pages copied by every lane of the producer
  using C = Cfg<FP8, P>;
  constexpr int NST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned (the TMA swizzle atom) by pointer arithmetic on the
  // shared array itself, so that every access below stays a shared-memory
  // access the compiler can tell apart from global memory
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = smem;
  float* comb = reinterpret_cast<float*>(smem + NST * C::kStageBytes);
  int2* plist = reinterpret_cast<int2*>(smem + NST * C::kStageBytes + C::kCombineBytes);
  int* pid = reinterpret_cast<int*>(plist + kWindow);                      // [kWindow] ids
  int4* meta = reinterpret_cast<int4*>(pid + kWindow);                     // [NST]
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + NST);
  uint64_t* empty = full + NST;
  uint64_t* cfull = empty + NST;           // the consumers' states are in comb
  uint64_t* cfree = cfull + 1;             // the merge warp is done reading comb
  uint64_t* cbar = cfree + 1;              // the consumer warps' barrier (last piece)
  int* wslot = reinterpret_cast<int*>(cbar + 1);                         // [NST] fetch mode
  __shared__ int s_abort;
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    mbar_init(cfull, kConsumerWarps);
    mbar_init(cfree, 1);
    mbar_init(cbar, kConsumerWarps);
    s_abort = 0;
    fence_barrier_init();
  }
  // the CTA's range, from the launch parameters alone: computed (and the
  // pages it will touch prefetched into L2, which also walks their address
  // translations) while the previous kernel drains
  const int t0 = tile_begin(p, cta), t1 = tile_begin(p, cta + 1);
  const int u_first = t0 / p.w, u_last = (t1 - 1) / p.w;
  if (warp == kProducerWarp) {
    if (lane == 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
    }
    const int row = u_first / p.Hkv;
    const void* pf = lane == 0   ? (const void*)(p.sel + (size_t)row * p.W)
                     : lane == 1 ? (const void*)(p.phys + (size_t)row * p.W)
                     : lane == 2 ? (const void*)(p.seq_lens + row % p.B)
                     : lane == 3 ? (const void*)(p.q + (size_t)u_first * p.G * kD)
                     : lane == 4 ? (const void*)(p.out + (size_t)u_first * p.G * kD)
                     : lane == 5 ? (const void*)(p.part_o + (size_t)cta * 2 * p.G * kD)
                     : lane == 6 ? (const void*)(p.part_ml + (size_t)cta * 2 * p.G * 2)
                                 : (const void*)(p.tickets + u_first);
    if (lane < 8) prefetch_l2(pf);
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();                 // sel, phys, q and the pool come from earlier kernels

  if (warp == kMergeWarp) {
    // ---------------- merge warp ---------------------------------------------
    // At the end of each piece but the CTA's last the consumers leave their
    // 4 softmax states in comb and stream on; this warp combines them: a
    // whole unit becomes its output, a shared unit's piece an (m, l, o)
    // partial, which it publishes (GPU-scope fence, atomic ticket).  The
    // last piece of a unit to arrive merges every piece into the output (a7).
    // The consumers finish the CTA's last piece themselves.
    const float* cO = comb;                                      // [4][8][D]
    const float* cM = cO + kConsumerWarps * kMaxG * kD;           // [4][8]
    const float* cL = cM + kConsumerWarps * kMaxG;                // [4][8]
    const int wl = lane >> 3, gl = lane & 7;      // lane = (warp, head) of the weights
    for (int u = u_first, k = 0; u < u_last; ++u, ++k) {
      if (!mbar_wait(cfull, k & 1, &s_abort)) {
        if (lane == 0) set_status(p.status, SSA_ST_TIMEOUT);
        return;
      }
      const int us = u * p.w;
      const int c_first = cta_of(p, us), c_last = cta_of(p, us + p.w - 1);
      const bool whole = c_first == c_last;
      const size_t pslot = (size_t)cta * 2 + (t0 >= us ? 0 : 1);
      // per head: M = max over the warps, the warps' factors, L
      const float mw = cM[wl * kMaxG + gl];
      float M = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 8));
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
      const float f = M == -INFINITY ? 0.0f : fast_exp2(mw - M);
      float L = cL[wl * kMaxG + gl] * f;
      L += __shfl_xor_sync(0xffffffffu, L, 8);
      L += __shfl_xor_sync(0xffffffffu, L, 16);
      __nv_bfloat16* outu = p.out + (size_t)u * p.G * kD;
#pragma unroll
      for (int gg = 0; gg < kMaxG; ++gg) {
        float fw[kConsumerWarps];
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) fw[w] = __shfl_sync(0xffffffffu, f, w * kMaxG + gg);
        const float Mg = __shfl_sync(0xffffffffu, M, gg), Lg = __shfl_sync(0xffffffffu, L, gg);
        if (gg >= p.G) continue;
        const float rL = Lg > 0.0f ? 1.0f / Lg : 0.0f;
#pragma unroll
        for (int i = 0; i < kD / 32; ++i) {
          const int d = lane + 32 * i, dz = d ^ (8 * ((gg >> 1) & 3));
          float O = 0.0f;
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) O += cO[(w * kMaxG + gg) * kD + dz] * fw[w];
          if (whole) outu[gg * kD + d] = __float2bfloat16_rn(O * rL);
          else p.part_o[(pslot * p.G + gg) * kD + d] = O;
        }
        if (!whole && lane == 0) {
          p.part_ml[(pslot * p.G + gg) * 2] = Mg;
          p.part_ml[(pslot * p.G + gg) * 2 + 1] = Lg;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(cfree);     // comb may take the next piece
      if (whole) continue;
      int last = 0;
      if (lane == 0) {
        __threadfence();
        last = atomicAdd(&p.tickets[u], 1) == c_last - c_first;
      }
      if (!__shfl_sync(0xffffffffu, last, 0)) continue;
      __threadfence();
      const int np = c_last - c_first + 1;
      const int slot0 = tile_begin(p, c_first) == us ? 0 : 1;
      // pieces: (c_first, slot0), then (c, 0) for c_first < c <= c_last
      auto piece = [&](int kk) -> size_t {
        return ((size_t)(c_first + kk) * 2 + (kk == 0 ? slot0 : 0)) * p.G;
      };
      // lane: d = 4*lane..4*lane+3 of every head; pieces in order
      const float2* pml = reinterpret_cast<const float2*>(p.part_ml);
      const float4* po = reinterpret_cast<const float4*>(p.part_o);
      float Mh[kMaxG], Lh[kMaxG];
      float4 acc[kMaxG];
#pragma unroll
      for (int jj = 0; jj < kMaxG; ++jj) {
        Mh[jj] = -INFINITY;
        Lh[jj] = 0.0f;
        acc[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int kk = 0; kk < np; ++kk) {      // a piece's vectors per round trip
        float2 ml[kMaxG];
        float4 x[kMaxG];
#pragma unroll
        for (int jj = 0; jj < kMaxG; ++jj) {
          ml[jj] = jj < p.G ? __ldcg(pml + piece(kk) + jj) : make_float2(-INFINITY, 0.0f);
          x[jj] = jj < p.G ? __ldcg(po + (piece(kk) + jj) * (kD / 4) + lane)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int jj = 0; jj < kMaxG; ++jj) merge_online(Mh[jj], Lh[jj], acc[jj], ml[jj], x[jj]);
      }
#pragma unroll
      for (int jj = 0; jj < kMaxG; ++jj) {
        if (jj < p.G) {
          const float r = Lh[jj] > 0.0f ? 1.0f / Lh[jj] : 0.0f;
          uint2 pk;
          pk.x = pack_bf16(acc[jj].x * r, acc[jj].y * r);
          pk.y = pack_bf16(acc[jj].z * r, acc[jj].w * r);
          *reinterpret_cast<uint2*>(outu + jj * kD + 4 * lane) = pk;
        }
      }
      if (lane == 0) p.tickets[u] = 0;       // ready for the next call
    }
    return;
  }

  if (warp == kProducerWarp) {
    // ---------------- producer warp ----------------------------------------
    // The warp reads and compacts the rows; lane 0 issues the TMA loads (the
    // resident path issues pages from lane 0 alone; the host-tail path from
    // the whole warp, every lane its share of 16-byte copies for a page
    // without a slot).  Lane 0's st counts the stages.  A stage's descriptor
    // carries it, and the consumers check it against the stage they waited
    // for.
    int st = 0;
    bool ok = true;
    int cur_row = -1, cnt = 0, seq_len = 0;
    int pgc[4], slc[4], idc[4];  // the row's first 128 entries, kept for the second pass

    auto acquire = [&](int s) -> bool {      // lane 0: stage slot s % NST is free
      return s < NST || mbar_wait(&empty[s % NST], ((s / NST) - 1) & 1, &s_abort);
    };
    auto acquire_warp = [&]() -> bool {
      bool acq = lane == 0 ? acquire(st) : true;
      return __shfl_sync(0xffffffffu, acq, 0);
    };
    auto issue_marker = [&](int kind, int unit) -> bool {   // the whole warp
      if (!acquire_warp()) return false;
      const int sb = st % NST;
      if (lane == 0) {
        meta[sb] = make_int4(kind, 0, unit, st);
        mbar_arrive(&full[sb]);
      }
      ++st;
      return true;
    };

    // one page of K and V (one KV head), its fp8 scales and, on the first
    // page of a piece, the unit's q rows.  Resident pages (ent.y >= 0, a
    // slot) come by TMA from the pool; pages from the host (ent.y <= -2: in
    // host-tail mode logical id -2 - ent.y; in fetch mode slot -2 - ent.y,
    // logical id mid) by 16-byte cp.async copies from the pinned mirror, every
    // lane a share, into the same swizzled stage layout, and in fetch mode
    // marked for the consumers to write into the slot.  The whole warp in
    // the host-tail and fetch modes, lane 0 alone in the resident mode.
    auto issue_page = [&](int2 ent, int mid, int flags, int unit, int h, int layer,
                          int seq_len) -> bool {
      if (!(WARP_ISSUE ? acquire_warp() : acquire(st))) return false;
      const int sb = st % NST;
      uint8_t* stage = ring + sb * C::kStageBytes;
      const uint32_t qbytes = (flags & kFirst) ? (uint32_t)p.G * kD * 2 : 0u;
      const bool host = WARP_ISSUE && ent.y < 0;
      if (FT && host) {
        flags |= kWriteBack;
        if (lane == 0) wslot[sb] = -2 - ent.y;
      }
      if constexpr (WARP_ISSUE) if (host) {
        const size_t id = (size_t)(FT ? mid : -2 - ent.y);
        const size_t pg_bytes = (size_t)p.Hkv * P * kD * (FP8 ? 1 : 2);
        const uint8_t* kpg = p.k_mir + ((size_t)layer * p.Lp + id) * pg_bytes;
        const uint8_t* vpg = p.v_mir + ((size_t)layer * p.Lp + id) * pg_bytes;
        const uint32_t sk = smem_u32(stage), sv = sk + C::kTileBytes;
        if (FP8) {
          // K rows [P][128 B] (128-byte swizzle); V d-rows [128][P B] (kVSwz)
          for (int i = lane; i < P * 8; i += 32) {
            const int t = i >> 3, uu = i & 7;
            cp_async16(sk + t * 128 + ((uu ^ (t & 7)) << 4),
                       kpg + ((size_t)(h * P + t) * 128 + uu * 16));
          }
          constexpr int kVu = P / 16;                      // 16-byte units per V row
          for (int i = lane; i < kD * kVu; i += 32) {
            const int d = i / kVu, uu = i - d * kVu;
            cp_async16(sv + swz(d * P + uu * 16, C::kVSwz),
                       vpg + ((size_t)(h * kD + d) * P + uu * 16));
          }
          const size_t so = ((size_t)layer * p.Lp + id) * P;
          for (int i = lane; i < 2 * (P / 4); i += 32) {
            const int which = i / (P / 4), uu = i - which * (P / 4);
            cp_async16(sk + 2 * C::kTileBytes + which * P * 4 + uu * 16,
                       (which ? p.vs_mir : p.ks_mir) + so + uu * 4);
          }
        } else {
          // K and V rows [P][256 B] as two 128-byte column halves, swizzled
          for (int i = lane; i < 2 * P * 16; i += 32) {
            const int which = i / (P * 16), r = i - which * P * 16;
            const int t = r >> 4, uu = r & 15, half = uu >> 3, u8 = uu & 7;
            cp_async16((which ? sv : sk) + half * (P * 128) + t * 128 + ((u8 ^ (t & 7)) << 4),
                       (which ? vpg : kpg) + ((size_t)(h * P + t) * 256 + uu * 16));
          }
        }
        cp_async_mbar_arrive(&full[sb]);
        __syncwarp();                          // every lane's copies are tracked first
      }
      if (lane == 0) {
        const int nvalid = max(0, min(P, seq_len - ent.x * P));
        meta[sb] = make_int4(flags, nvalid, unit, st);
        mbar_arrive_expect_tx(&full[sb],
                              (host ? 0u : (uint32_t)(2 * C::kTileBytes + C::kScaleBytes)) + qbytes);
        if (!host) {
          const int row_k = ((layer * p.S + ent.y) * p.Hkv + h) * P;
          if (FP8) {
            tma_load_2d(stage, &tmK, &full[sb], 0, row_k);
            const int row_v = ((layer * p.S + ent.y) * p.Hkv + h) * kD;
            tma_load_2d(stage + C::kTileBytes, &tmV, &full[sb], 0, row_v);
            const size_t so = ((size_t)layer * p.S + ent.y) * P;
            bulk_load(stage + 2 * C::kTileBytes, p.k_scale + so, P * 4, &full[sb]);
            bulk_load(stage + 2 * C::kTileBytes + P * 4, p.v_scale + so, P * 4, &full[sb]);
          } else {
            tma_load_2d(stage, &tmK, &full[sb], 0, row_k);
            tma_load_2d(stage + P * 128, &tmK, &full[sb], 64, row_k);
            tma_load_2d(stage + C::kTileBytes, &tmV, &full[sb], 0, row_k);
            tma_load_2d(stage + C::kTileBytes + P * 128, &tmV, &full[sb], 64, row_k);
          }
        }
        if (qbytes) bulk_load(stage + C::kQOff, p.q + (size_t)unit * p.G * kD, qbytes, &full[sb]);
      }
      ++st;
      return true;
    };

    for (int u = u_first; u <= u_last && ok; ++u) {
      const int us = u * p.w;
      const int a = max(t0, us) - us;
      const int e = min(t1, us + p.w) - us;
      const int row = u / p.Hkv, h = u - row * p.Hkv;
      const int li = row / p.B, b = row - li * p.B;
      const int layer = p.layer0 + li;
      const int32_t* selr = p.sel + (size_t)row * p.W;
      const int32_t* physr = HT ? nullptr : p.phys + (size_t)row * p.W;
      auto phys_at = [&](int i) -> int { return physr ? physr[i] : -1; };
      // host tail: the slot of each selected page from slot_of; a page with
      // no slot is encoded as -2 - (its logical id) and read from the mirror;
      // an out-of-range id as S (flagged, skipped)
      auto resolve = [&](int (&pg)[4], int (&sl)[4]) {
        int id[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          id[k] = pg[k] >= 0 && pg[k] < p.nmax ? p.bt[(size_t)b * p.nmax + pg[k]] : -1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const bool ok_id = id[k] >= 0 && id[k] < p.Lp;
          const int slot = ok_id ? p.slot_of[(size_t)layer * p.Lp + id[k]] : -1;
          sl[k] = !ok_id ? (pg[k] >= 0 ? p.S : -1) : (slot >= 0 ? slot : -2 - id[k]);
        }
      };
      // fetch mode: the logical ids of the marked entries (pages to fetch);
      // an out-of-range id marks the entry S (flagged, skipped)
      auto resolve_ids = [&](const int (&pg)[4], int (&sl)[4], int (&id)[4]) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          id[k] = sl[k] <= -2 && pg[k] >= 0 && pg[k] < p.nmax ? p.bt[(size_t)b * p.nmax + pg[k]]
                                                              : -1;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (sl[k] <= -2 && (id[k] < 0 || id[k] >= p.Lp || -2 - sl[k] >= p.S)) sl[k] = p.S;
      };
      auto entry_valid = [&](int pg_, int sl_) -> bool {
        return pg_ >= 0 && ((sl_ >= 0 && sl_ < p.S) || (WARP_ISSUE && sl_ <= -2));
      };
      if (row != cur_row) {      // count the row's valid entries (once per row)
        cur_row = row;
        seq_len = p.seq_lens[b];
        cnt = 0;
        for (int base = 0; base < p.W; base += 4 * 32) {
          int pg[4], sl[4], id[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {        // every load of the batch in flight at once
            const int i = base + 32 * k + lane;
            pg[k] = i < p.W ? selr[i] : -1;
            sl[k] = i < p.W ? phys_at(i) : -1;
          }
          if (HT) resolve(pg, sl);
          if (FT) resolve_ids(pg, sl, id);
          if (base == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) { pgc[k] = pg[k]; slc[k] = sl[k]; idc[k] = FT ? id[k] : -1; }
          }
          int bad = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const bool valid = entry_valid(pg[k], sl[k]);
            if (pg[k] >= 0 && sl[k] >= p.S) bad |= SSA_ST_BAD_ID;
            else if (pg[k] >= 0 && !valid) bad |= SSA_ST_UNRESOLVED;
            cnt += __popc(__ballot_sync(0xffffffffu, valid));
          }
          if (bad) set_status(p.status, bad);
        }
      }
      // this piece's share [a, e) of the unit's weight, as valid entries [j0, j1)
      const int j0 = (int)((long long)a * cnt / p.w), j1 = (int)((long long)e * cnt / p.w);
      if (j0 == j1) {
        ok = issue_marker(kEmpty | (u == u_last ? kFinal : 0), u);
        continue;
      }
      int seen = 0, issued = 0;
      for (int base = 0; base < p.W && seen < j1 && ok; base += 4 * 32) {
        int pgv[4], slv[4], idv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = base + 32 * k + lane;
          pgv[k] = base == 0 ? pgc[k] : (i < p.W ? selr[i] : -1);
          slv[k] = base == 0 ? slc[k] : (i < p.W ? phys_at(i) : -1);
          idv[k] = base == 0 ? idc[k] : -1;
        }
        if (HT && base > 0) resolve(pgv, slv);
        if (FT && base > 0) resolve_ids(pgv, slv, idv);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (seen >= j1 || !ok) break;
          const bool valid = entry_valid(pgv[k], slv[k]);
          const unsigned lt = (1u << lane) - 1u;
          const unsigned m = __ballot_sync(0xffffffffu, valid);
          const int rank = seen + __popc(m & lt);
          const bool in = valid && rank >= j0 && rank < j1;
          const unsigned mi = __ballot_sync(0xffffffffu, in);
          if (in) {
            plist[__popc(mi & lt)] = make_int2(pgv[k], slv[k]);
            pid[__popc(mi & lt)] = idv[k];
          }
          __syncwarp();
          const int nw = __popc(mi);
          if (WARP_ISSUE || lane == 0) {       // the resident path issues from lane 0 alone
            for (int x = 0; x < nw && ok; ++x, ++issued) {
              const int flags = (issued == 0 ? kFirst : 0) |
                                (issued == j1 - j0 - 1 ? (u == u_last ? kLast | kFinal : kLast) : 0);
              ok = issue_page(plist[x], pid[x], flags, u, h, layer, seq_len);
            }
          }
          if (!WARP_ISSUE) ok = __shfl_sync(0xffffffffu, ok, 0);
          __syncwarp();                        // the window is rewritten next round
          seen += __popc(m);
        }
      }
    }
    if (ok) ok = issue_marker(kDone, 0);
    if (lane != 0) return;
    if (!ok) {
      s_abort = 1;
      set_status(p.status, SSA_ST_TIMEOUT);
      // let every copy still in flight land before the CTA can exit
      for (int s = st > NST ? st - NST : 0; s < st; ++s)
        mbar_wait(&full[s % NST], (s / NST) & 1, nullptr);
    }
    return;
  }

  // ---------------- consumers -------------------------------------------------
  // QK^T: A = 16 K rows (tokens), B = q^T (8 heads), C = S^T[token][head].
  // PV:   A = V^T rows (16 of d), B = P^T (C transposed in registers by
  //       movmatrix), C = O^T[d][head].  No MMA row is padding.
  const int r4 = lane >> 2, c = lane & 3;

  uint32_t qb[8][2];
  float qscale_log2 = p.sm_log2;
  float o[8][4];   // O^T: rows d = 16*mt + r4 (+8), columns (heads) 2c, 2c+1
  // softmax state of heads 2c, 2c+1 (the lanes that own those O^T columns);
  // fp8: probabilities carry v_scale / vref, vref a power of two above every
  // V scale seen so far (0 before the first block)
  float m_run0, m_run1, l_run0, l_run1, vref;
  auto reset = [&]() {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
    m_run0 = m_run1 = -INFINITY;
    l_run0 = l_run1 = 0.0f;
    vref = FP8 ? 0.0f : 1.0f;
  };
  reset();
  // token of MMA row r4 and r4+8 within a 16-token block.  fp8: rows 2j, 2j+1
  // and 2j+8, 2j+9 are the 4 consecutive tokens 4j..4j+3 that one 32-bit
  // word of a V d-row holds, in order, so the word converts straight into
  // the PV fragment.  (Two of a K ldmatrix's 8 rows then share a swizzle
  // chunk, a 2-way bank conflict; swapping pairs to avoid it cost a shift
  // per V word and measured slower.)
  int tauA = r4, tauB = r4 + 8;
  if (FP8) {
    const int j = r4 >> 1, e = r4 & 1;
    tauA = 4 * j + e;
    tauB = 4 * j + 2 + e;
  }
  // fp8: the MMA fragments come from ldmatrix, lane i giving the address of
  // row i & 7 of matrix i >> 3.  QK, per k32 step: (rows tauA, chunk 2ks),
  // (rows tauB, 2ks), (tauA, 2ks + 1), (tauB, 2ks + 1) -- each lane gets the
  // 4 bytes at 4c of row r4, as one 32-bit read per fragment did.  PV, per
  // pair of 16-row d tiles: d rows 0-7 and 8-15 of the first tile, then of
  // the second, 16 tokens each.
  uint32_t kq_row = 0, kq_c0 = 0, kq_sw = 0, v_row = 0;
  if (FP8) {
    const int mi = lane >> 3, rr = lane & 7;
    const int jj = rr >> 1, ee = rr & 1;
    const int tA = 4 * jj + ee, tB = 4 * jj + 2 + ee;
    const int t = (mi & 1) ? tB : tA;
    kq_row = (uint32_t)t * 128;
    kq_sw = (uint32_t)(t & 7);
    kq_c0 = (uint32_t)(mi >> 1);
    v_row = (uint32_t)(16 * (mi >> 1) + 8 * (mi & 1) + rr);
  }

  // End of a piece: leave this warp's state in comb for the merge warp
  // (once it has read the previous piece's) and stream on.  The consumer
  // warps never wait for one another.
  int n_flush = 0;
  auto flush = [&]() -> bool {
    float l0 = l_run0, l1 = l_run1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    if (n_flush > 0 && !mbar_wait(cfree, (n_flush - 1) & 1, &s_abort)) return false;
    float* cO = comb;                                             // [4][8][D]
    float* cM = cO + kConsumerWarps * kMaxG * kD;                  // [4][8]
    float* cL = cM + kConsumerWarps * kMaxG;                       // [4][8]
    // row (warp, head g) of cO holds column d at d ^ (8 * ((g >> 1) & 3)):
    // the 32 lanes of a store (heads 2c, columns r4 + 16 mt) hit 32 banks
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d = (16 * mt + r4) ^ (8 * c);
      cO[(warp * kMaxG + 2 * c) * kD + d] = o[mt][0] * vref;
      cO[(warp * kMaxG + 2 * c + 1) * kD + d] = o[mt][1] * vref;
      cO[(warp * kMaxG + 2 * c) * kD + (d ^ 8)] = o[mt][2] * vref;
      cO[(warp * kMaxG + 2 * c + 1) * kD + (d ^ 8)] = o[mt][3] * vref;
    }
    if (r4 == 0) {
      cM[warp * kMaxG + 2 * c] = m_run0;
      cM[warp * kMaxG + 2 * c + 1] = m_run1;
      cL[warp * kMaxG + 2 * c] = l0;
      cL[warp * kMaxG + 2 * c + 1] = l1;
    }
    reset();
    __syncwarp();
    if (lane == 0) mbar_arrive(cfull);
    ++n_flush;
    return true;
  };

  // The CTA's last piece: the consumer warps combine, publish and, when
  // they hold the unit's last piece, merge it themselves (the merge warp is
  // done by then; they would otherwise sit idle).
  uint32_t cph = 0;
  auto csync = [&]() -> bool {             // one arrival per warp, bounded wait
    __syncwarp();
    if (lane == 0) mbar_arrive(cbar);
    const bool ok = mbar_wait(cbar, cph, &s_abort);
    cph ^= 1u;
    return ok;
  };
  auto final_flush = [&](int unit) -> bool {
    float l0 = l_run0, l1 = l_run1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    if (n_flush > 0 && !mbar_wait(cfree, (n_flush - 1) & 1, &s_abort)) return false;
    float* cO = comb;
    float* cM = cO + kConsumerWarps * kMaxG * kD;
    float* cL = cM + kConsumerWarps * kMaxG;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d = (16 * mt + r4) ^ (8 * c);
      cO[(warp * kMaxG + 2 * c) * kD + d] = o[mt][0] * vref;
      cO[(warp * kMaxG + 2 * c + 1) * kD + d] = o[mt][1] * vref;
      cO[(warp * kMaxG + 2 * c) * kD + (d ^ 8)] = o[mt][2] * vref;
      cO[(warp * kMaxG + 2 * c + 1) * kD + (d ^ 8)] = o[mt][3] * vref;
    }
    if (r4 == 0) {
      cM[warp * kMaxG + 2 * c] = m_run0;
      cM[warp * kMaxG + 2 * c + 1] = m_run1;
      cL[warp * kMaxG + 2 * c] = l0;
      cL[warp * kMaxG + 2 * c + 1] = l1;
    }
    if (!csync()) return false;
    const int us = unit * p.w;
    const int c_first = cta_of(p, us), c_last = cta_of(p, us + p.w - 1);
    const bool whole = c_first == c_last;
    const size_t pslot = (size_t)cta * 2 + (t0 >= us ? 0 : 1);
    __nv_bfloat16* outu = p.out + (size_t)unit * p.G * kD;
    // thread tid owns column d = tid of every head: 8 independent chains
    const int d = tid;
#pragma unroll
    for (int gg = 0; gg < kMaxG; ++gg) {
      if (gg < p.G) {
        const int dz = d ^ (8 * ((gg >> 1) & 3));
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cM[w * kMaxG + gg]);
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float f = fast_exp2(cM[w * kMaxG + gg] - M);
            L += cL[w * kMaxG + gg] * f;
            O += cO[(w * kMaxG + gg) * kD + dz] * f;
          }
        }
        if (whole) {
          outu[gg * kD + d] = __float2bfloat16_rn(O * (L > 0.0f ? 1.0f / L : 0.0f));
        } else {
          const size_t pi = pslot * p.G + gg;
          p.part_o[pi * kD + d] = O;
          if (d == 0) {
            p.part_ml[pi * 2] = M;
            p.part_ml[pi * 2 + 1] = L;
          }
        }
      }
    }
    if (whole) return true;
    // publish: every partial write of the CTA, then one GPU-scope fence and
    // the ticket
    if (!csync()) return false;
    if (tid == 0) {
      __threadfence();
      s_last = atomicAdd(&p.tickets[unit], 1) == c_last - c_first;
    }
    if (!csync()) return false;
    if (!s_last) return true;
    __threadfence();
    const int np = c_last - c_first + 1;
    const int slot0 = tile_begin(p, c_first) == us ? 0 : 1;
    auto piece = [&](int kk) -> size_t {
      return ((size_t)(c_first + kk) * 2 + (kk == 0 ? slot0 : 0)) * p.G;
    };
    // thread: d = 4*lane..+3 of heads warp and warp + 4; the same merge as
    // the merge warp's (merge_online in piece order), four pieces' loads per
    // round trip (a unit rarely spans more than four CTAs)
    const float2* pml = reinterpret_cast<const float2*>(p.part_ml);
    const float4* po = reinterpret_cast<const float4*>(p.part_o);
    float Mh[2] = {-INFINITY, -INFINITY}, Lh[2] = {0.0f, 0.0f};
    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    constexpr int kMB = 4;
    for (int k0 = 0; k0 < np; k0 += kMB) {
      float2 ml[kMB][2];
      float4 x[kMB][2];
#pragma unroll
      for (int kk = 0; kk < kMB; ++kk)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int g = warp + 4 * hh;
          const bool ok = k0 + kk < np && g < p.G;
          ml[kk][hh] = ok ? __ldcg(pml + piece(k0 + kk) + g) : make_float2(-INFINITY, 0.0f);
          x[kk][hh] = ok ? __ldcg(po + (piece(k0 + kk) + g) * (kD / 4) + lane)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int kk = 0; kk < kMB; ++kk)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) merge_online(Mh[hh], Lh[hh], acc[hh], ml[kk][hh], x[kk][hh]);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int g = warp + 4 * hh;
      if (g < p.G) {
        const float r = Lh[hh] > 0.0f ? 1.0f / Lh[hh] : 0.0f;
        uint2 pk;
        pk.x = pack_bf16(acc[hh].x * r, acc[hh].y * r);
        pk.y = pack_bf16(acc[hh].z * r, acc[hh].w * r);
        *reinterpret_cast<uint2*>(outu + g * kD + 4 * lane) = pk;
      }
    }
    if (tid == 0) p.tickets[unit] = 0;     // ready for the next call
    return true;
  };

  // One call site for each flush, so that its code exists once.
  int pc = 0;                              // pages processed
  for (int st = 0;; ++st) {
    int fkind = 0, funit = u_last;         // 1 = flush, 2 = final_flush
    {
      const int sb = st % NST;
      if (!mbar_wait(&full[sb], (st / NST) & 1, &s_abort)) {
        s_abort = 1;
        set_status(p.status, SSA_ST_TIMEOUT);
        break;
      }
      const int4 dsc = meta[sb];
      if (dsc.w != st) {                   // not the stage this warp waited for
        s_abort = 1;
        set_status(p.status, SSA_ST_INTERNAL);
        break;
      }
      if (dsc.x & kDone) break;
      if (dsc.x & kEmpty) {
        if (lane == 0) mbar_arrive(&empty[sb]);
        fkind = (dsc.x & kFinal) ? 2 : 1;
        funit = dsc.z;
        goto flushes;
      }
      const int nvalid = dsc.y;
      uint8_t* stage = ring + sb * C::kStageBytes;
      const uint32_t kb = smem_u32(stage);
      const uint32_t vb = kb + C::kTileBytes;
      const float* ksc = reinterpret_cast<const float*>(stage + 2 * C::kTileBytes);
      const float* vsc = ksc + P;

      if (dsc.x & kFirst) {
        // the unit's G query rows as the B operand (rows >= G are zero).
        // bf16: b0 = q[r4][k 2c, 2c+1], b1 = q[r4][k 2c+8, 2c+9] per k16 step.
        // fp8: q * 2^eq as two e4m3 terms hi + lo (the top and the next four
        // significant bits: their sum is q * 2^eq to within 2^-10, i.e.
        // ~2^-18 of |q|max), so QK runs as e4m3 MMAs on the raw K codes;
        // per k32 step b0 = d 32ks + 4c..+3, b1 = d + 16; qb[ks] = hi,
        // qb[4 + ks] = lo
        const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(stage + C::kQOff);
        const bool row_ok = r4 < p.G;
        if (FP8) {
          float amax = 0.0f;
          for (int i = lane; i < p.G * (kD / 8); i += 32)
            amax = fmaxf(amax, bf16x8_absmax(*reinterpret_cast<const uint4*>(qs + i * 8)));
          amax = warp_max(amax);
          int eq = 0;
          if (amax > 0.0f) {
            const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFF);   // amax in [2^(ef-127), 2^(ef-126))
            eq = 134 - ef;                                                // amax * 2^eq in [128, 256)
            eq = eq > 126 ? 126 : (eq < -126 ? -126 : eq);
          }
          const float up = exp2f((float)eq);
          qscale_log2 = p.sm_log2 * exp2f((float)-eq);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const __nv_bfloat16* r = qs + r4 * kD + 32 * ks + 16 * half + 4 * c;
              float x[4], y[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) x[i] = row_ok ? __bfloat162float(r[i]) * up : 0.0f;
              const uint32_t hi = f32x4_to_e4m3x4(x[0], x[1], x[2], x[3]);
              e4m3x4_to_f32x4(hi, y[0], y[1], y[2], y[3]);
              qb[ks][half] = hi;
              qb[4 + ks][half] = f32x4_to_e4m3x4(x[0] - y[0], x[1] - y[1], x[2] - y[2], x[3] - y[3]);
            }
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            qb[ks][0] = row_ok ? *reinterpret_cast<const uint32_t*>(qs + r4 * kD + 16 * ks + 2 * c) : 0u;
            qb[ks][1] = row_ok ? *reinterpret_cast<const uint32_t*>(qs + r4 * kD + 16 * ks + 2 * c + 8) : 0u;
          }
        }
      }

      // NB 16-token blocks per warp step share one softmax update (max,
      // rescale, V-scale reference) and interleave their MMA chains.  Two per
      // step measured no faster than one on GB300 and needs more registers
      // than two CTAs per SM leave, so one.
      constexpr int NB = 1;
      constexpr int kSteps = C::kBlocks / NB;
      // this warp's blocks of the page: the stream's block index
      // pc * kSteps + bs taken round-robin, block bs == warp - pc*kSteps mod 4
#pragma unroll 1
      for (int bs = (warp - pc * kSteps) & (kConsumerWarps - 1); bs < kSteps;
           bs += kConsumerWarps) {
        const int tb0 = bs * NB * 16;
        if (FT && (dsc.x & kWriteBack)) {
          // fetch mode: this block's rows of the fetched page go to its slot
          // (before any zeroing below), K, V and, from KV head 0, the scales
          const int slot = wslot[sb];
          const int row = dsc.z / p.Hkv, hh = dsc.z - row * p.Hkv;
          const int layer = p.layer0 + row / p.B;
          const size_t hp = ((size_t)layer * p.S + slot) * p.Hkv + hh;      // head-page index
          if (FP8) {
            uint8_t* kp = p.k_pool + hp * (P * kD);                        // [P][128]
            uint8_t* vp = p.v_pool + hp * (P * kD);                        // [128][P]
            for (int i = lane; i < NB * 16 * 8; i += 32) {
              const int r = tb0 + (i >> 3), uu = i & 7;
              *reinterpret_cast<uint4*>(kp + r * 128 + uu * 16) =
                  *reinterpret_cast<const uint4*>(stage + r * 128 + ((uu ^ (r & 7)) << 4));
            }
            for (int i = lane; i < kD * NB; i += 32) {
              const int d = i / NB, j = i - d * NB;
              *reinterpret_cast<uint4*>(vp + d * P + tb0 + 16 * j) =
                  *reinterpret_cast<const uint4*>(stage + C::kTileBytes +
                                                  swz(d * P + tb0 + 16 * j, C::kVSwz));
            }
            if (hh == 0 && lane < 8 * NB) {
              const int which = lane / (4 * NB), uu = lane - which * 4 * NB;
              float* dst = const_cast<float*>(which ? p.v_scale : p.k_scale) +
                           ((size_t)layer * p.S + slot) * P;
              *reinterpret_cast<uint4*>(dst + tb0 + uu * 4) = *reinterpret_cast<const uint4*>(
                  stage + 2 * C::kTileBytes + which * P * 4 + (tb0 + uu * 4) * 4);
            }
          } else {
            uint8_t* kp = p.k_pool + hp * (P * kD * 2);                    // [P][256 B]
            uint8_t* vp = p.v_pool + hp * (P * kD * 2);
            for (int i = lane; i < 2 * NB * 16 * 16; i += 32) {
              const int which = i / (NB * 256), rr = i - which * NB * 256;
              const int r = tb0 + (rr >> 4), uu = rr & 15, half = uu >> 3, u8 = uu & 7;
              *reinterpret_cast<uint4*>((which ? vp : kp) + r * 256 + uu * 16) =
                  *reinterpret_cast<const uint4*>(stage + which * C::kTileBytes + half * (P * 128) +
                                                  r * 128 + ((u8 ^ (r & 7)) << 4));
            }
          }
        }
        // zero V of the tokens past seq_len (their bytes are not ours to trust)
        if (nvalid < tb0 + NB * 16) {
          for (int j = 0; j < NB; ++j) {
            const int tb = tb0 + 16 * j;
            if (nvalid >= tb + 16) continue;
            if (FP8) {
              for (int i = lane; i < kD * 16; i += 32) {
                const int d = i >> 4, xx = tb + (i & 15);
                if (xx >= nvalid) stage[C::kTileBytes + swz(d * P + xx, C::kVSwz)] = 0;
              }
            } else {
              for (int i = lane; i < 16 * 16; i += 32) {
                const int r = tb + (i >> 4), ch = i & 15;
                if (r >= nvalid)
                  *reinterpret_cast<uint4*>(stage + C::kTileBytes + (ch >> 3) * (P * 128) +
                                            r * 128 + (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
              }
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
        }

        // S^T = K q^T per block; rows: x[j][0], x[j][1] = token tkA[j], heads
        // 2c, 2c+1; x[j][2], x[j][3] = token tkB[j]
        float x[NB][4], vsA[NB], vsB[NB];
        int tkA[NB], tkB[NB];
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          const int tb = tb0 + 16 * j;
          float s4[4] = {0.f, 0.f, 0.f, 0.f}, sx[4] = {0.f, 0.f, 0.f, 0.f};
          tkA[j] = tb + tauA;
          tkB[j] = tb + tauB;
          if (FP8) {
            // A = the K codes as they are: a0/a2 = token tkA, d 32ks + 4c..+3
            // and d + 16; a1/a3 = token tkB.  hi and lo terms in two chains.
            // The block's rows start at a multiple of 16 tokens, so a row's
            // swizzle (token & 7) is the lane's constant kq_sw.
            const uint32_t kr = kb + (uint32_t)tb * 128 + kq_row;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4(a0, a1, a2, a3, kr + (((2 * ks + kq_c0) ^ kq_sw) << 4));
              mma_e4m3(s4, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
              mma_e4m3(sx, a0, a1, a2, a3, qb[4 + ks][0], qb[4 + ks][1]);
            }
          } else {
            const int mi = lane >> 3, rr = lane & 7;
            const int t = tb + (mi & 1) * 8 + rr;
            const uint32_t rowk = kb + t * 128;
            const int xt = t & 7;
#pragma unroll
            for (int ks = 0; ks < 8; ks += 2) {
              uint32_t a0, a1, a2, a3, a4, a5, a6, a7;
              const int c0 = 2 * ks + (mi >> 1), c1 = c0 + 2;     // 16-byte chunks over d
              ldsm_x4(a0, a1, a2, a3, rowk + (c0 >> 3) * (P * 128) + (((c0 & 7) ^ xt) << 4));
              ldsm_x4(a4, a5, a6, a7, rowk + (c1 >> 3) * (P * 128) + (((c1 & 7) ^ xt) << 4));
              mma_bf16(s4, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
              mma_bf16(sx, a4, a5, a6, a7, qb[ks + 1][0], qb[ks + 1][1]);
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) x[j][i] = (s4[i] + sx[i]) * qscale_log2;
          vsA[j] = vsB[j] = 0.0f;
          if (FP8) {
            const float kA = ksc[tkA[j]], kB = ksc[tkB[j]];
            x[j][0] *= kA; x[j][1] *= kA; x[j][2] *= kB; x[j][3] *= kB;
            vsA[j] = vsc[tkA[j]];
            vsB[j] = vsc[tkB[j]];
          }
          if (nvalid < tb + 16) {          // the tail of a request's last page
            if (tkA[j] >= nvalid) { x[j][0] = x[j][1] = -INFINITY; vsA[j] = 0.0f; }
            if (tkB[j] >= nvalid) { x[j][2] = x[j][3] = -INFINITY; vsB[j] = 0.0f; }
          }
        }
        // The running maximum is a reference, not the exact maximum: it moves
        // only when a score of the step exceeds it by more than 2^kSlack, so
        // the probabilities stay below 2^kSlack (inside the f16 and bf16
        // operand ranges).  Only then are the exact per-head maxima reduced
        // over the 8 lanes r4 = 0..7 of c; after the first blocks most steps
        // skip the shuffles.  The same holds for the fp8 V-scale reference.
        float mx0 = fmaxf(x[0][0], x[0][2]), mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
        for (int j = 1; j < NB; ++j) {
          mx0 = fmaxf(mx0, fmaxf(x[j][0], x[j][2]));
          mx1 = fmaxf(mx1, fmaxf(x[j][1], x[j][3]));
        }
        float mn0 = m_run0, mn1 = m_run1, corr0 = 1.0f, corr1 = 1.0f;
        if (__any_sync(0xffffffffu, mx0 > m_run0 + kSlack || mx1 > m_run1 + kSlack)) {
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          mn0 = fmaxf(m_run0, mx0);
          mn1 = fmaxf(m_run1, mx1);
          corr0 = fast_exp2(m_run0 - (mn0 == -INFINITY ? 0.0f : mn0));
          corr1 = fast_exp2(m_run1 - (mn1 == -INFINITY ? 0.0f : mn1));
        }
        const float mu0 = mn0 == -INFINITY ? 0.0f : mn0, mu1 = mn1 == -INFINITY ? 0.0f : mn1;
        float oc0 = corr0, oc1 = corr1;
        float vinv = 1.0f;
        if (FP8) {
          float vmax = fmaxf(vsA[0], vsB[0]);
#pragma unroll
          for (int j = 1; j < NB; ++j) vmax = fmaxf(vmax, fmaxf(vsA[j], vsB[j]));
          if (__any_sync(0xffffffffu, vmax >= vref)) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1)
              vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
            // every lane holds the same tokens' scales: vmax is the step's
            const float nref = __uint_as_float(((__float_as_uint(vmax) >> 23) + 1) << 23);
            const float ratio = vref * pow2_rcp(nref);
            oc0 *= ratio;
            oc1 *= ratio;
            vref = nref;
          }
          vinv = pow2_rcp(vref);
        }
        uint32_t b0[NB], b1[NB];
        float ls0 = 0.0f, ls1 = 0.0f;
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          const float p0 = fast_exp2(x[j][0] - mu0), p1 = fast_exp2(x[j][1] - mu1);
          const float p2 = fast_exp2(x[j][2] - mu0), p3 = fast_exp2(x[j][3] - mu1);
          uint32_t P0, P1;
          if (FP8) {
            ls0 += p0 + p2;
            ls1 += p1 + p3;
            const float wA = vsA[j] * vinv, wB = vsB[j] * vinv;
            P0 = pack_f16(p0 * wA, p1 * wA);
            P1 = pack_f16(p2 * wB, p3 * wB);
          } else {
            const float q0 = bf16_round(p0), q1 = bf16_round(p1);
            const float q2 = bf16_round(p2), q3 = bf16_round(p3);
            ls0 += q0 + q2;
            ls1 += q1 + q3;
            P0 = pack_bf16(q0, q1);
            P1 = pack_bf16(q2, q3);
          }
          // P^T as the B operand: each 8x8 half transposed across the warp
          b0[j] = movmatrix_trans(P0);
          b1[j] = movmatrix_trans(P1);
        }
        l_run0 = l_run0 * corr0 + ls0;
        l_run1 = l_run1 * corr1 + ls1;
        m_run0 = mn0;
        m_run1 = mn1;
        if (__any_sync(0xffffffffu, oc0 != 1.0f || oc1 != 1.0f)) {
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            o[mt][0] *= oc0; o[mt][1] *= oc1; o[mt][2] *= oc0; o[mt][3] *= oc1;
          }
        }

        // O^T += V^T P^T, 16 rows of d per MMA, the step's blocks in turn
        if (FP8) {
          // rows d = 16*mt + r4 and +8, one ldmatrix per two tiles: the
          // swizzle bits do not depend on the tile (32*P per pair is a
          // multiple of the swizzle period), so the lane's address is
          // computed once per block
#pragma unroll
          for (int j = 0; j < NB; ++j) {
            const uint32_t va = vb + swz(v_row * P + tb0 + 16 * j, C::kVSwz);
#pragma unroll
            for (int mp = 0; mp < 4; ++mp) {
              uint32_t w[4];             // tile 2mp rows r4, r4 + 8; tile 2mp + 1 the same
              ldsm_x4(w[0], w[1], w[2], w[3], va + mp * 32 * P);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t a0, a1, a2, a3;
                e4m3x4_to_f16x2x2(w[2 * h], a0, a2);
                e4m3x4_to_f16x2x2(w[2 * h + 1], a1, a3);
                mma_f16(o[2 * mp + h], a0, a1, a2, a3, b0[j], b1[j]);
              }
            }
          }
        } else {
          const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
            for (int j = 0; j < NB; ++j) {
              const int t = tb0 + 16 * j + (mi >> 1) * 8 + rr;
              const int chunk = 2 * mt + (mi & 1);
              const uint32_t addr =
                  vb + (chunk >> 3) * (P * 128) + t * 128 + (((chunk & 7) ^ (t & 7)) << 4);
              uint32_t a0, a1, a2, a3;
              ldsm_x4_t(a0, a1, a2, a3, addr);
              mma_bf16(o[mt], a0, a1, a2, a3, b0[j], b1[j]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[sb]);
      ++pc;
      if (dsc.x & kLast) {
        fkind = (dsc.x & kFinal) ? 2 : 1;
        funit = dsc.z;
      }
    }
  flushes:
    if (fkind == 1 && !flush()) break;
    if (fkind == 2 && !final_flush(funit)) break;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool make_tmap(CUtensorMap* tm, void* base, CUtensorMapDataType dt, int esz, uint64_t inner,
               uint64_t rows, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * (uint64_t)esz};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FP8, int P>
size_t decode_smem() {
  using C = Cfg<FP8, P>;
  return 1024 + (size_t)C::kStages * C::kStageBytes + C::kCombineBytes + kWindow * 12 +
         (size_t)C::kStages * 16 + 2 * C::kStages * 8 + 4 * 8 + (size_t)C::kStages * 4;
}

// CTAs of one wave: resident CTAs per SM (the configuration's target, or
// what the occupancy calculator grants, whichever is lower) x SMs, cut so
// that every CTA gets at least four tiles and no unit more than 130 pieces
// (a small launch split over fewer, longer ranges merges fewer pieces per
// unit: 27.3 -> 21.2 us for 24 units of 33 pages, the same for larger ones).
template <bool FP8, int P, int MODE>
int decode_grid(const Dims& d, int n_layers, int num_sms) {
  // per device: the occupancy calculator's answer depends on the GPU
  static std::atomic<int> occ_of[kMaxDevices];
  std::atomic<int>& slot = occ_of[current_device_ordinal()];
  int occ = slot.load(std::memory_order_relaxed);
  if (occ < 1) {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, decode_kernel<FP8, P, MODE>,
                                                      kDecodeThreads,
                                                      decode_smem<FP8, P>()) != cudaSuccess)
      o = 1;
    occ = o < 1 ? 1 : (o > Cfg<FP8, P>::kCtasPerSm ? Cfg<FP8, P>::kCtasPerSm : o);
    slot.store(occ, std::memory_order_relaxed);
  }
  const int w = d.max_selected();
  const long long T = (long long)n_layers * d.B * d.Hkv * w;
  const int tpc_min = w > 256 ? (w + 127) / 128 : 4;
  long long n = T / tpc_min;
  if (n > (long long)num_sms * occ) n = (long long)num_sms * occ;
  return n < 1 ? 1 : (int)n;
}

template <bool FP8, int P, int MODE>
cudaError_t launch_decode_t(const DecodeArgs& a, DecodeParams& p, cudaStream_t s) {
  const Dims& d = *a.d;
  const ssa_cache& c = *a.c;
  CUtensorMap tmK, tmV;
  const uint64_t rows_tok = (uint64_t)d.Lyr * d.S * d.Hkv * P;
  bool ok;
  if (FP8) {
    ok = make_tmap(&tmK, c.k_pool, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kD, rows_tok, kD, P,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    const CUtensorMapSwizzle vsw = P >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : P == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                                 : P == 32  ? CU_TENSOR_MAP_SWIZZLE_32B
                                            : CU_TENSOR_MAP_SWIZZLE_NONE;
    ok = ok && make_tmap(&tmV, c.v_pool, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, P,
                         (uint64_t)d.Lyr * d.S * d.Hkv * kD, P, kD, vsw);
  } else {
    ok = make_tmap(&tmK, c.k_pool, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, rows_tok, 64, P,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_tmap(&tmV, c.v_pool, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, rows_tok, 64, P,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!ok) return cudaErrorInvalidValue;
  const size_t smem = decode_smem<FP8, P>();
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<FP8, P, MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int n = decode_grid<FP8, P, MODE>(d, a.n_layers, a.num_sms);
  if (n > decode_max_ctas(d, a.num_sms)) return cudaErrorInvalidValue;   // workspace bound
  p.w = d.max_selected();
  const long long T = (long long)a.n_layers * d.B * d.Hkv * p.w;
  if (T > INT_MAX / 2) return cudaErrorInvalidValue;
  p.T = (int)T;
  p.tq = p.T / n;
  p.tr = p.T % n;
  e = launch_pdl(decode_kernel<FP8, P, MODE>, dim3(n), dim3(kDecodeThreads), smem, s, p, tmK,
                 tmV);
  count_launch();
  return e;
}

}  // namespace

int decode_ctas_per_sm(const Dims& d) {
  switch (d.P * 2 + d.fp8) {
    case 32: return Cfg<false, 16>::kCtasPerSm;
    case 33: return Cfg<true, 16>::kCtasPerSm;
    case 64: return Cfg<false, 32>::kCtasPerSm;
    case 65: return Cfg<true, 32>::kCtasPerSm;
    case 128: return Cfg<false, 64>::kCtasPerSm;
    case 129: return Cfg<true, 64>::kCtasPerSm;
    case 256: return Cfg<false, 128>::kCtasPerSm;
    default: return Cfg<true, 128>::kCtasPerSm;
  }
}

int decode_max_ctas(const Dims& d, int num_sms) { return num_sms * decode_ctas_per_sm(d); }

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  const Dims& d = *a.d;
  const ssa_cache& c = *a.c;
  DecodeParams p{};
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.sel = a.sel;
  p.phys = a.phys;
  p.seq_lens = a.seq_lens;
  p.k_scale = c.k_scale;
  p.v_scale = c.v_scale;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.part_o = a.part_o;
  p.part_ml = a.part_ml;
  p.tickets = a.tickets;
  p.status = a.status;
  p.layer0 = a.layer0;
  p.B = d.B; p.Hq = d.Hq; p.Hkv = d.Hkv; p.G = d.G; p.W = d.W; p.S = d.S;
  p.sm_log2 = a.sm_scale * 1.4426950408889634f;
  p.host_tail = a.host_tail;
  p.k_pool = static_cast<uint8_t*>(c.k_pool);
  p.v_pool = static_cast<uint8_t*>(c.v_pool);
  p.Lp = d.Lp;
  p.nmax = d.nmax;
  p.bt = a.bt;
  p.slot_of = c.slot_of;
  p.k_mir = static_cast<const uint8_t*>(c.k_mirror);
  p.v_mir = static_cast<const uint8_t*>(c.v_mirror);
  p.ks_mir = c.k_scale_mirror;
  p.vs_mir = c.v_scale_mirror;
  const int mode = a.fetch ? kFetch : (a.host_tail ? kHostTail : kResident);
  switch ((d.P * 2 + d.fp8) * 4 + mode) {
    case 128: return launch_decode_t<false, 16, 0>(a, p, s);
    case 129: return launch_decode_t<false, 16, 1>(a, p, s);
    case 130: return launch_decode_t<false, 16, 2>(a, p, s);
    case 132: return launch_decode_t<true, 16, 0>(a, p, s);
    case 133: return launch_decode_t<true, 16, 1>(a, p, s);
    case 134: return launch_decode_t<true, 16, 2>(a, p, s);
    case 256: return launch_decode_t<false, 32, 0>(a, p, s);
    case 257: return launch_decode_t<false, 32, 1>(a, p, s);
    case 258: return launch_decode_t<false, 32, 2>(a, p, s);
    case 260: return launch_decode_t<true, 32, 0>(a, p, s);
    case 261: return launch_decode_t<true, 32, 1>(a, p, s);
    case 262: return launch_decode_t<true, 32, 2>(a, p, s);
    case 512: return launch_decode_t<false, 64, 0>(a, p, s);
    case 513: return launch_decode_t<false, 64, 1>(a, p, s);
    case 514: return launch_decode_t<false, 64, 2>(a, p, s);
    case 516: return launch_decode_t<true, 64, 0>(a, p, s);
    case 517: return launch_decode_t<true, 64, 1>(a, p, s);
    case 518: return launch_decode_t<true, 64, 2>(a, p, s);
    case 1024: return launch_decode_t<false, 128, 0>(a, p, s);
    case 1025: return launch_decode_t<false, 128, 1>(a, p, s);
    case 1026: return launch_decode_t<false, 128, 2>(a, p, s);
    case 1028: return launch_decode_t<true, 128, 0>(a, p, s);
    case 1029: return launch_decode_t<true, 128, 1>(a, p, s);
    case 1030: return launch_decode_t<true, 128, 2>(a, p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssa
