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
//     movmatrix), m16n8k16 tensor-core tiles, fp32 accumulate, online softmax
//     in the log2 domain with warp shuffles;
//   * bf16 K/V: bf16 MMAs, ldmatrix (V transposed by ldmatrix.trans);
//   * fp8 K/V: the e4m3 codes convert exactly to f16, so the MMAs run in f16
//     on the raw codes; q is scaled by a power of two into f16 range, the K
//     scale multiplies the fp32 score, and the V scale folds into the
//     probabilities (relative to a running power-of-two reference, so the
//     f16 operand never overflows).  V is stored d-major in the pool
//     ([Hkv][D][P]) so that the 8-bit reads run along tokens, the reduction
//     axis of PV;
//   * at the end of a piece each consumer warp leaves its softmax state in
//     shared memory and streams on; a sixth warp combines the 4 states: a
//     whole unit becomes its output, a shared unit's piece an (m, l, o)
//     partial that it publishes (GPU-scope fence, atomic ticket); the last
//     piece of a unit to arrive merges the unit's partials into the output.
//     No CTA ever waits for another, no consumer warp for another.
// The work is HBM-bound (8 flop/byte bf16, 16 fp8): the tensor cores carry
// the G-row tiles, the memory system sets the pace.
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
constexpr int kSmemPerSm = 228 * 1024;
constexpr int kSmemPerCtaMax = 227 * 1024;
constexpr int kSmemReservedPerCta = 1024;

// stage descriptor flags
constexpr int kQ = 1;       // the stage also holds the unit's q rows
constexpr int kFlush = 2;   // no data: the end of a piece (one such stage per consumer warp)
constexpr int kDone = 4;    // no data: the end of the CTA's range (one per consumer warp)
constexpr int kSeqShift = 4;  // the descriptor's flags word holds the chunk index above this

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

// A stage holds one chunk: up to kCT tokens of one page of one KV head (K and
// V tiles, fp8 scales) and, for a consumer warp's first chunk of a unit, the
// unit's q rows.  One consumer warp processes a whole chunk (kNB 16-token
// blocks, their MMA chains interleaved); chunk j of the CTA's stream goes to
// consumer warp j % 4 and stage j % kStages (a multiple of 4, so each stage
// serves one warp).
template <bool FP8, int P>
struct Cfg {
  static constexpr int kCT = FP8 ? (P < 64 ? P : 64) : (P < 32 ? P : 32);   // tokens per chunk
  static constexpr int kChunks = P / kCT;                                     // chunks per page
  static constexpr int kNB = kCT / 16;                                        // blocks per chunk
  static constexpr int kTileBytes = kCT * kD * (FP8 ? 1 : 2);    // K (or V) of one chunk
  static constexpr int kScaleBytes = FP8 ? 2 * kCT * 4 : 0;
  static constexpr int kQOff = 2 * kTileBytes + kScaleBytes;
  static constexpr int kQBytes = kMaxG * kD * 2;
  static constexpr int kStageBytes = round_up(kQOff + kQBytes, 1024);
  static constexpr int kCombineBytes = kConsumerWarps * kMaxG * kD * 4 + 2 * kConsumerWarps * kMaxG * 4;
  // alignment slack, combine area, producer window, descriptors and barriers
  static constexpr int kFixed = 1024 + kCombineBytes + kWindow * 8 + kMaxStages * 32 + 64;
  // two CTAs per SM when at least four stages fit beside the second CTA
  static constexpr int kStages2 = (kSmemPerSm / 2 - kSmemReservedPerCta - kFixed) / kStageBytes;
  static constexpr int kCtasPerSm = kStages2 >= 4 ? 2 : 1;
  static constexpr int kStagesFit =
      kCtasPerSm == 2 ? kStages2 : (kSmemPerCtaMax - kFixed) / kStageBytes;
  // a multiple of the consumer warps: chunk j takes stage j % kStages and goes
  // to warp j % 4, so every stage belongs to one warp, and a warp's wait on a
  // stage's barrier parity always follows its own wait on the previous phase
  static constexpr int kStages =
      (kStagesFit > kMaxStages ? kMaxStages : kStagesFit) / kConsumerWarps * kConsumerWarps;
  // log2 of the fp8 V^T row swizzle span in 16-byte units (row = kCT bytes)
  static constexpr int kVSwz = kCT >= 128 ? 3 : (kCT == 64 ? 2 : (kCT == 32 ? 1 : 0));
  static_assert(kStages >= kConsumerWarps && kStages % kConsumerWarps == 0,
                "whole stages per consumer warp");
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

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
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

// First tile of CTA c (the first tr CTAs hold tq + 1 tiles, the others
// tq), and the CTA that holds tile t (the inverse).
__device__ __forceinline__ int tile_begin(const DecodeParams& p, int c) {
  return c * p.tq + min(c, p.tr);
}
__device__ __forceinline__ int cta_of(const DecodeParams& p, int t) {
  const int big = p.tr * (p.tq + 1);
  return t < big ? t / (p.tq + 1) : p.tr + (t - big) / p.tq;
}

template <bool FP8, int P>
__global__ void __launch_bounds__(kDecodeThreads, Cfg<FP8, P>::kCtasPerSm)
decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV) {
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
  int4* meta = reinterpret_cast<int4*>(plist + kWindow);                  // [NST]
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + NST);
  uint64_t* empty = full + NST;
  uint64_t* cfull = empty + NST;           // the consumers' states are in comb
  uint64_t* cfree = cfull + 1;             // the merge warp is done reading comb
  uint64_t* cbar = cfree + 1;              // the consumer warps' barrier (last piece)
  __shared__ int s_abort;
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);           // the one consumer warp of the chunk
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
      // lane g < G: running max and sum of head g over the pieces
      float Mu = -INFINITY, Lu = 0.0f;
      if (lane < p.G) {
#pragma unroll 4
        for (int kk = 0; kk < np; ++kk) {
          const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + piece(kk) + lane);
          if (ml.x > Mu) {
            Lu *= fast_exp2(Mu - ml.x);
            Mu = ml.x;
          }
          if (ml.x != -INFINITY) Lu += ml.y * fast_exp2(ml.x - Mu);
        }
      }
      const float invL = Lu > 0.0f ? 1.0f / Lu : 0.0f;
      // lane holds d = 4*lane..4*lane+3 of every head; a piece's weight
      // comes from its head's lane
      const float4* po = reinterpret_cast<const float4*>(p.part_o);
      float4 acc[kMaxG];
#pragma unroll
      for (int jj = 0; jj < kMaxG; ++jj) acc[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int kk = 0; kk < np; ++kk) {      // a piece's vectors per round trip
        float f = 0.0f;
        if (lane < p.G && Mu != -INFINITY)
          f = fast_exp2(__ldcg(&p.part_ml[(piece(kk) + lane) * 2]) - Mu);
        float4 x[kMaxG];
#pragma unroll
        for (int jj = 0; jj < kMaxG; ++jj)
          x[jj] = jj < p.G ? __ldcg(po + (piece(kk) + jj) * (kD / 4) + lane)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int jj = 0; jj < kMaxG; ++jj) {
          const float wj = __shfl_sync(0xffffffffu, f, jj);
          acc[jj].x += wj * x[jj].x; acc[jj].y += wj * x[jj].y;
          acc[jj].z += wj * x[jj].z; acc[jj].w += wj * x[jj].w;
        }
      }
#pragma unroll
      for (int jj = 0; jj < kMaxG; ++jj) {
        const float r = __shfl_sync(0xffffffffu, invL, jj);
        if (jj < p.G) {
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
    // The warp reads and compacts the rows; lane 0 alone issues the copies.
    // Chunks go out in range order: chunk st to stage st % NST, for consumer
    // warp st % 4.  The first four chunks of a piece carry the unit's q rows
    // (they reach four different warps, so every warp that gets any chunk of
    // the piece gets q with its first one).  After each piece but the CTA's
    // last come four kFlush stages, one per consumer warp, and after the last
    // piece four kDone stages: a warp ends its piece on its marker, which
    // depends on no stage issued later (so no warp waits, holding a stage,
    // for a flush that needs a stage not yet issued).
    constexpr int CT = C::kCT;
    int st = 0;                 // chunks issued (every lane keeps the count)
    bool ok = true;
    int cur_row = -1, cnt = 0, seq_len = 0;
    int pgc[4], slc[4];        // the row's first 128 entries, kept for the second pass

    auto acquire = [&](int s) -> bool {      // lane 0: stage slot s % NST is free
      return s < NST || mbar_wait(&empty[s % NST], ((s / NST) - 1) & 1, &s_abort);
    };
    // meta.x: the flags and, above them, the chunk's index in the stream
    // (the consumer checks it against the index it waited for).  Called by
    // the whole warp; st advances in every lane.
    auto issue_marker = [&](int kind, int piece) -> bool {
      bool acq = lane == 0 ? acquire(st) : true;
      acq = __shfl_sync(0xffffffffu, acq, 0);
      if (!acq) return false;
      const int sb = st % NST;
      if (lane == 0) {
        meta[sb] = make_int4(kind | (st << kSeqShift), 0, 0, piece);
        mbar_arrive(&full[sb]);
      }
      ++st;
      return true;
    };

    // chunk ci of one page of K and V (one KV head), its fp8 scales and,
    // with kQ, the unit's q rows.  Resident pages (ent.y >= 0, a slot) come
    // by TMA from the pool; host-tail pages (ent.y <= -2, logical id
    // -2 - ent.y) by 16-byte cp.async copies from the pinned mirror, every
    // lane a share, into the same swizzled stage layout.  Called by the
    // whole warp.
    auto issue_chunk = [&](int2 ent, int ci, int flags, int unit, int piece, int h, int layer,
                           int seq_len) -> bool {
      bool acq = lane == 0 ? acquire(st) : true;
      acq = __shfl_sync(0xffffffffu, acq, 0);
      if (!acq) return false;
      const int sb = st % NST;
      uint8_t* stage = ring + sb * C::kStageBytes;
      const uint32_t qbytes = (flags & kQ) ? (uint32_t)p.G * kD * 2 : 0u;
      const bool host = ent.y < 0;
      if (host) {
        const size_t id = (size_t)(-2 - ent.y);
        const size_t pg_bytes = (size_t)p.Hkv * P * kD * (FP8 ? 1 : 2);
        const uint8_t* kpg = p.k_mir + ((size_t)layer * p.Lp + id) * pg_bytes;
        const uint8_t* vpg = p.v_mir + ((size_t)layer * p.Lp + id) * pg_bytes;
        const uint32_t sk = smem_u32(stage), sv = sk + C::kTileBytes;
        if (FP8) {
          // K rows [CT][128 B] (128-byte swizzle); V d-rows [128][CT B] (kVSwz)
          for (int i = lane; i < CT * 8; i += 32) {
            const int t = i >> 3, uu = i & 7;
            cp_async16(sk + t * 128 + ((uu ^ (t & 7)) << 4),
                       kpg + ((size_t)(h * P + ci * CT + t) * 128 + uu * 16));
          }
          constexpr int kVu = CT / 16;                     // 16-byte units per V row
          for (int i = lane; i < kD * kVu; i += 32) {
            const int d = i / kVu, uu = i - d * kVu;
            cp_async16(sv + swz(d * CT + uu * 16, C::kVSwz),
                       vpg + ((size_t)(h * kD + d) * P + ci * CT + uu * 16));
          }
          const size_t so = ((size_t)layer * p.Lp + id) * P + ci * CT;
          for (int i = lane; i < 2 * (CT / 4); i += 32) {
            const int which = i / (CT / 4), uu = i - which * (CT / 4);
            cp_async16(sk + 2 * C::kTileBytes + which * CT * 4 + uu * 16,
                       (which ? p.vs_mir : p.ks_mir) + so + uu * 4);
          }
        } else {
          // K and V rows [CT][256 B] as two 128-byte column halves, swizzled
          for (int i = lane; i < 2 * CT * 16; i += 32) {
            const int which = i / (CT * 16), r = i - which * CT * 16;
            const int t = r >> 4, uu = r & 15, half = uu >> 3, u8 = uu & 7;
            cp_async16((which ? sv : sk) + half * (CT * 128) + t * 128 + ((u8 ^ (t & 7)) << 4),
                       (which ? vpg : kpg) + ((size_t)(h * P + ci * CT + t) * 256 + uu * 16));
          }
        }
        cp_async_mbar_arrive(&full[sb]);
        __syncwarp();                          // every lane's copies are tracked first
      }
      if (lane == 0) {
        const int nvalid = max(0, min(CT, seq_len - ent.x * P - ci * CT));
        meta[sb] = make_int4(flags | (st << kSeqShift), nvalid, unit, piece);
        mbar_arrive_expect_tx(&full[sb],
                              (host ? 0u : (uint32_t)(2 * C::kTileBytes + C::kScaleBytes)) + qbytes);
        if (!host) {
          const int row_k = ((layer * p.S + ent.y) * p.Hkv + h) * P + ci * CT;
          if (FP8) {
            tma_load_2d(stage, &tmK, &full[sb], 0, row_k);
            const int row_v = ((layer * p.S + ent.y) * p.Hkv + h) * kD;
            tma_load_2d(stage + C::kTileBytes, &tmV, &full[sb], ci * CT, row_v);
            const size_t so = ((size_t)layer * p.S + ent.y) * P + ci * CT;
            bulk_load(stage + 2 * C::kTileBytes, p.k_scale + so, CT * 4, &full[sb]);
            bulk_load(stage + 2 * C::kTileBytes + CT * 4, p.v_scale + so, CT * 4, &full[sb]);
          } else {
            tma_load_2d(stage, &tmK, &full[sb], 0, row_k);
            tma_load_2d(stage + CT * 128, &tmK, &full[sb], 64, row_k);
            tma_load_2d(stage + C::kTileBytes, &tmV, &full[sb], 0, row_k);
            tma_load_2d(stage + C::kTileBytes + CT * 128, &tmV, &full[sb], 64, row_k);
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
      const int piece = u - u_first;
      const int32_t* selr = p.sel + (size_t)row * p.W;
      const int32_t* physr = p.host_tail ? nullptr : p.phys + (size_t)row * p.W;
      auto physr_or_null = [&](int i) -> int { return physr ? physr[i] : -1; };
      // host tail: the slot of each selected page from slot_of; a page with
      // no slot is encoded as -2 - (its logical id) and read from the mirror
      auto resolve = [&](int (&pg)[4], int (&sl)[4], int layer_, int b_) {
        int id[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          id[k] = pg[k] >= 0 && pg[k] < p.nmax ? p.bt[(size_t)b_ * p.nmax + pg[k]] : -1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const bool ok_id = id[k] >= 0 && id[k] < p.Lp;
          const int slot = ok_id ? p.slot_of[(size_t)layer_ * p.Lp + id[k]] : -1;
          sl[k] = !ok_id ? (pg[k] >= 0 ? p.S : -1) : (slot >= 0 ? slot : -2 - id[k]);
        }
      };
      auto entry_valid = [&](int pg_, int sl_) -> bool {
        return pg_ >= 0 && ((sl_ >= 0 && sl_ < p.S) || (p.host_tail && sl_ <= -2));
      };
      if (row != cur_row) {      // count the row's valid entries (once per row)
        cur_row = row;
        seq_len = p.seq_lens[b];
        cnt = 0;
        for (int base = 0; base < p.W; base += 4 * 32) {
          int pg[4], sl[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {        // every load of the batch in flight at once
            const int i = base + 32 * k + lane;
            pg[k] = i < p.W ? selr[i] : -1;
            sl[k] = i < p.W ? physr_or_null(i) : -1;
          }
          if (p.host_tail) resolve(pg, sl, layer, b);
          if (base == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) { pgc[k] = pg[k]; slc[k] = sl[k]; }
          }
          int bad = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const bool valid = entry_valid(pg[k], sl[k]);
            if (pg[k] >= 0 && sl[k] < 0 && !valid && sl[k] != p.S) bad |= SSA_ST_UNRESOLVED;
            if (pg[k] >= 0 && sl[k] >= p.S) bad |= SSA_ST_BAD_ID;
            cnt += __popc(__ballot_sync(0xffffffffu, valid));
          }
          if (bad) set_status(p.status, bad);
        }
      }
      // this piece's share [a, e) of the unit's weight, as valid entries [j0, j1)
      const int j0 = (int)((long long)a * cnt / p.w), j1 = (int)((long long)e * cnt / p.w);
      int seen = j0 == j1 ? p.W : 0, issued = 0;      // no pages: markers only
      for (int base = 0; base < p.W && seen < j1 && ok; base += 4 * 32) {
        int pgv[4], slv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = base + 32 * k + lane;
          pgv[k] = base == 0 ? pgc[k] : (i < p.W ? selr[i] : -1);
          slv[k] = base == 0 ? slc[k] : (i < p.W ? physr_or_null(i) : -1);
        }
        if (base > 0 && p.host_tail) resolve(pgv, slv, layer, b);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (seen >= j1 || !ok) break;
          const bool valid = entry_valid(pgv[k], slv[k]);
          const unsigned lt = (1u << lane) - 1u;
          const unsigned m = __ballot_sync(0xffffffffu, valid);
          const int rank = seen + __popc(m & lt);
          const bool in = valid && rank >= j0 && rank < j1;
          const unsigned mi = __ballot_sync(0xffffffffu, in);
          if (in) plist[__popc(mi & lt)] = make_int2(pgv[k], slv[k]);
          __syncwarp();
          const int nw = __popc(mi);
          for (int x = 0; x < nw && ok; ++x) {
            const int2 ent = plist[x];
            for (int ci = 0; ci < C::kChunks && ok; ++ci) {
              if (ci > 0 && ent.x * P + ci * CT >= seq_len) break;   // past the request's end
              ok = issue_chunk(ent, ci, issued < kConsumerWarps ? kQ : 0, u, piece, h, layer,
                               seq_len);
              ++issued;
            }
          }
          __syncwarp();                        // the window is rewritten next round
          seen += __popc(m);
        }
      }
      if (u < u_last)
        for (int i = 0; i < kConsumerWarps && ok; ++i) ok = issue_marker(kFlush, piece);
    }
    for (int i = 0; i < kConsumerWarps && ok; ++i) ok = issue_marker(kDone, u_last - u_first);
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
  // Each consumer warp takes whole chunks (chunk j of the CTA's stream when
  // j % 4 == warp), the kNB 16-token blocks of a chunk in one pass with their
  // MMA chains interleaved and one softmax update per chunk.
  // QK^T: A = 16 K rows (tokens), B = q^T (8 heads), C = S^T[token][head].
  // PV:   A = V^T rows (16 of d), B = P^T (C transposed in registers by
  //       movmatrix), C = O^T[d][head].  No MMA row is padding.
  constexpr int CT = C::kCT;
  constexpr int NB = C::kNB;
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
  const int rot = c >= 2 ? 16 : 0;      // fp8 V: lanes 2, 3 hold the token pairs swapped
  // token of MMA row r4 and r4+8 within a 16-token block.  fp8: rows 2j, 2j+1
  // and 2j+8, 2j+9 cover the 4 consecutive tokens 4j..4j+3 that one 32-bit V
  // read returns, lanes of j >= 2 taking the pairs swapped so that the 8 rows
  // one K read touches fall in distinct swizzle chunks (no bank conflicts)
  int tauA = r4, tauB = r4 + 8;
  if (FP8) {
    const int j = r4 >> 1, e = r4 & 1;
    tauA = 4 * j + (j < 2 ? e : 2 + e);
    tauB = 4 * j + (j < 2 ? 2 + e : e);
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
    // thread: d = 4*lane..+3 of heads warp and warp + 4; online merge of the
    // pieces, two pieces' loads per round trip
    const float2* pml = reinterpret_cast<const float2*>(p.part_ml);
    const float4* po = reinterpret_cast<const float4*>(p.part_o);
    float Mh[2] = {-INFINITY, -INFINITY}, Lh[2] = {0.0f, 0.0f};
    float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int k0 = 0; k0 < np; k0 += 2) {
      float2 ml[2][2];
      float4 x[2][2];
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int g = warp + 4 * hh;
          const bool ok = k0 + kk < np && g < p.G;
          ml[kk][hh] = ok ? __ldcg(pml + piece(k0 + kk) + g) : make_float2(-INFINITY, 0.0f);
          x[kk][hh] = ok ? __ldcg(po + (piece(k0 + kk) + g) * (kD / 4) + lane)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float m = ml[kk][hh].x;
          if (m == -INFINITY) continue;
          const float mn = fmaxf(Mh[hh], m);
          const float a = fast_exp2(Mh[hh] - mn), b = fast_exp2(m - mn);
          Lh[hh] = Lh[hh] * a + ml[kk][hh].y * b;
          acc[hh].x = acc[hh].x * a + x[kk][hh].x * b;
          acc[hh].y = acc[hh].y * a + x[kk][hh].y * b;
          acc[hh].z = acc[hh].z * a + x[kk][hh].z * b;
          acc[hh].w = acc[hh].w * a + x[kk][hh].w * b;
          Mh[hh] = mn;
        }
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

  // The chunk stream: a warp ends a piece on its kFlush stage (its state,
  // possibly empty, goes to the merge warp) and the CTA's last piece on its
  // kDone stage.
  bool done = false;
  for (int j = warp;; j += kConsumerWarps) {
    const int sb = j % NST;
    if (!mbar_wait(&full[sb], (j / NST) & 1, &s_abort)) {
      s_abort = 1;
      set_status(p.status, SSA_ST_TIMEOUT);
      break;
    }
    const int4 dsc = meta[sb];
    if ((dsc.x >> kSeqShift) != j) {        // not the chunk this warp waited for
      s_abort = 1;
      set_status(p.status, SSA_ST_INTERNAL);
      break;
    }
    if (dsc.x & kDone) {
      if (lane == 0) mbar_arrive(&empty[sb]);
      done = true;
      break;
    }
    if (dsc.x & kFlush) {
      const bool ok = flush();
      if (lane == 0) mbar_arrive(&empty[sb]);
      if (!ok) break;
      continue;
    }
    const int nvalid = dsc.y;
    uint8_t* stage = ring + sb * C::kStageBytes;
    const uint32_t kb = smem_u32(stage);
    const uint32_t vb = kb + C::kTileBytes;
    const float* ksc = reinterpret_cast<const float*>(stage + 2 * C::kTileBytes);
    const float* vsc = ksc + CT;

    if (dsc.x & kQ) {
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

    // zero V of the tokens past seq_len (their bytes are not ours to trust)
    if (nvalid < CT) {
      if (FP8) {
        for (int i = lane; i < kD * CT; i += 32) {
          const int d = i / CT, xx = i - d * CT;
          if (xx >= nvalid) stage[C::kTileBytes + swz(d * CT + xx, C::kVSwz)] = 0;
        }
      } else {
        for (int i = lane; i < CT * 16; i += 32) {
          const int r = i >> 4, ch = i & 15;
          if (r >= nvalid)
            *reinterpret_cast<uint4*>(stage + C::kTileBytes + (ch >> 3) * (CT * 128) + r * 128 +
                                      (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }

    // S^T = K q^T, the chunk's NB blocks side by side; block j rows:
    // x[j][0], x[j][1] = token 16j + tauA, heads 2c, 2c+1; x[j][2], x[j][3] =
    // token 16j + tauB
    float x[NB][4], vsA[NB], vsB[NB];
    {
      // fp8: one accumulator chain per block (the NB blocks give NB
      // independent chains); bf16: two per block (even and odd k steps)
      constexpr int NX = FP8 ? 1 : NB;
      float s4[NB][4], sx[NX][4];
#pragma unroll
      for (int jb = 0; jb < NB; ++jb)
#pragma unroll
        for (int i = 0; i < 4; ++i) s4[jb][i] = 0.0f;
#pragma unroll
      for (int jb = 0; jb < NX; ++jb)
#pragma unroll
        for (int i = 0; i < 4; ++i) sx[jb][i] = 0.0f;
      if (FP8) {
        // A = the K codes as they are: a0/a2 = token tkA, d 32ks + 4c..+3 and
        // d + 16; a1/a3 = token tkB.  The hi and lo terms accumulate in turn.
        const int xA = tauA & 7, xB = tauB & 7;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
          for (int jb = 0; jb < NB; ++jb) {
            const uint32_t rA = kb + (16 * jb + tauA) * 128 + 4 * c;
            const uint32_t rB = kb + (16 * jb + tauB) * 128 + 4 * c;
            const uint32_t a0 = lds32(rA + (((2 * ks) ^ xA) << 4));
            const uint32_t a1 = lds32(rB + (((2 * ks) ^ xB) << 4));
            const uint32_t a2 = lds32(rA + (((2 * ks + 1) ^ xA) << 4));
            const uint32_t a3 = lds32(rB + (((2 * ks + 1) ^ xB) << 4));
            mma_e4m3(s4[jb], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
            mma_e4m3(s4[jb], a0, a1, a2, a3, qb[4 + ks][0], qb[4 + ks][1]);
          }
        }
      } else {
        const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
        for (int ks = 0; ks < 8; ks += 2) {
#pragma unroll
          for (int jb = 0; jb < NB; ++jb) {
            const int t = 16 * jb + (mi & 1) * 8 + rr;
            const uint32_t rowk = kb + t * 128;
            const int xt = t & 7;
            uint32_t a0, a1, a2, a3, a4, a5, a6, a7;
            const int c0 = 2 * ks + (mi >> 1), c1 = c0 + 2;     // 16-byte chunks over d
            ldsm_x4(a0, a1, a2, a3, rowk + (c0 >> 3) * (CT * 128) + (((c0 & 7) ^ xt) << 4));
            ldsm_x4(a4, a5, a6, a7, rowk + (c1 >> 3) * (CT * 128) + (((c1 & 7) ^ xt) << 4));
            mma_bf16(s4[jb], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
            mma_bf16(sx[FP8 ? 0 : jb], a4, a5, a6, a7, qb[ks + 1][0], qb[ks + 1][1]);
          }
        }
      }
#pragma unroll
      for (int jb = 0; jb < NB; ++jb) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          x[jb][i] = (FP8 ? s4[jb][i] : s4[jb][i] + sx[FP8 ? 0 : jb][i]) * qscale_log2;
        const int tkA = 16 * jb + tauA, tkB = 16 * jb + tauB;
        vsA[jb] = vsB[jb] = 0.0f;
        if (FP8) {
          const float kA = ksc[tkA], kB = ksc[tkB];
          x[jb][0] *= kA; x[jb][1] *= kA; x[jb][2] *= kB; x[jb][3] *= kB;
          vsA[jb] = vsc[tkA];
          vsB[jb] = vsc[tkB];
        }
        if (nvalid < CT) {                // the tail of a request's last page
          if (tkA >= nvalid) { x[jb][0] = x[jb][1] = -INFINITY; vsA[jb] = 0.0f; }
          if (tkB >= nvalid) { x[jb][2] = x[jb][3] = -INFINITY; vsB[jb] = 0.0f; }
        }
      }
    }
    // per-head maxima over the chunk's tokens: the 8 lanes r4 = 0..7 of c
    float mx0 = fmaxf(x[0][0], x[0][2]), mx1 = fmaxf(x[0][1], x[0][3]);
#pragma unroll
    for (int jb = 1; jb < NB; ++jb) {
      mx0 = fmaxf(mx0, fmaxf(x[jb][0], x[jb][2]));
      mx1 = fmaxf(mx1, fmaxf(x[jb][1], x[jb][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m_run0, mx0), mn1 = fmaxf(m_run1, mx1);
    const float mu0 = mn0 == -INFINITY ? 0.0f : mn0, mu1 = mn1 == -INFINITY ? 0.0f : mn1;
    const float corr0 = fast_exp2(m_run0 - mu0), corr1 = fast_exp2(m_run1 - mu1);
    float oc0 = corr0, oc1 = corr1;
    float vinv = 1.0f;
    if (FP8) {
      float vmax = fmaxf(vsA[0], vsB[0]);
#pragma unroll
      for (int jb = 1; jb < NB; ++jb) vmax = fmaxf(vmax, fmaxf(vsA[jb], vsB[jb]));
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
        vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
      if (vmax >= vref) {
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
    for (int jb = 0; jb < NB; ++jb) {
      const float p0 = fast_exp2(x[jb][0] - mu0), p1 = fast_exp2(x[jb][1] - mu1);
      const float p2 = fast_exp2(x[jb][2] - mu0), p3 = fast_exp2(x[jb][3] - mu1);
      uint32_t P0, P1;
      if (FP8) {
        ls0 += p0 + p2;
        ls1 += p1 + p3;
        const float wA = vsA[jb] * vinv, wB = vsB[jb] * vinv;
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
      b0[jb] = movmatrix_trans(P0);
      b1[jb] = movmatrix_trans(P1);
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

    // O^T += V^T P^T, 16 rows of d per MMA; per row tile the chunk's blocks
    if (FP8) {
      // rows d = 16*mt + r4 and +8: the swizzle bits do not depend on mt
      // (16*CT*mt is a multiple of the swizzle period), so hoist them
      uint32_t va0[NB], va1[NB];
#pragma unroll
      for (int jb = 0; jb < NB; ++jb) {
        va0[jb] = vb + swz(r4 * CT + 16 * jb + 4 * c, C::kVSwz);
        va1[jb] = vb + swz((r4 + 8) * CT + 16 * jb + 4 * c, C::kVSwz);
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
        for (int jb = 0; jb < NB; ++jb) {
          uint32_t w0 = lds32(va0[jb] + mt * 16 * CT);
          uint32_t w1 = lds32(va1[jb] + mt * 16 * CT);
          w0 = __funnelshift_l(w0, w0, rot);
          w1 = __funnelshift_l(w1, w1, rot);
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(w0, a0, a2);
          e4m3x4_to_f16x2x2(w1, a1, a3);
          mma_f16(o[mt], a0, a1, a2, a3, b0[jb], b1[jb]);
        }
      }
    } else {
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
        for (int jb = 0; jb < NB; ++jb) {
          const int t = 16 * jb + (mi >> 1) * 8 + rr;
          const int chunk = 2 * mt + (mi & 1);
          const uint32_t addr =
              vb + (chunk >> 3) * (CT * 128) + t * 128 + (((chunk & 7) ^ (t & 7)) << 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(a0, a1, a2, a3, addr);
          mma_bf16(o[mt], a0, a1, a2, a3, b0[jb], b1[jb]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[sb]);
  }
  if (done) final_flush(u_last);
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
  return 1024 + (size_t)C::kStages * C::kStageBytes + C::kCombineBytes + kWindow * 8 +
         (size_t)C::kStages * 16 + 2 * C::kStages * 8 + 4 * 8;
}

// CTAs of one wave: resident CTAs per SM (the configuration's target, or
// what the occupancy calculator grants, whichever is lower) x SMs, cut so
// that every CTA gets at least two tiles and no unit more than 130 pieces.
template <bool FP8, int P>
int decode_grid(const Dims& d, int n_layers, int num_sms) {
  // per device: the occupancy calculator's answer depends on the GPU
  static std::atomic<int> occ_of[kMaxDevices];
  std::atomic<int>& slot = occ_of[current_device_ordinal()];
  int occ = slot.load(std::memory_order_relaxed);
  if (occ < 1) {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, decode_kernel<FP8, P>, kDecodeThreads,
                                                      decode_smem<FP8, P>()) != cudaSuccess)
      o = 1;
    occ = o < 1 ? 1 : (o > Cfg<FP8, P>::kCtasPerSm ? Cfg<FP8, P>::kCtasPerSm : o);
    slot.store(occ, std::memory_order_relaxed);
  }
  const int w = d.max_selected();
  const long long T = (long long)n_layers * d.B * d.Hkv * w;
  const int tpc_min = w > 256 ? (w + 127) / 128 : 2;
  long long n = T / tpc_min;
  if (n > (long long)num_sms * occ) n = (long long)num_sms * occ;
  return n < 1 ? 1 : (int)n;
}

template <bool FP8, int P>
cudaError_t launch_decode_t(const DecodeArgs& a, DecodeParams& p, cudaStream_t s) {
  const Dims& d = *a.d;
  const ssa_cache& c = *a.c;
  CUtensorMap tmK, tmV;
  const uint64_t rows_tok = (uint64_t)d.Lyr * d.S * d.Hkv * P;
  bool ok;
  constexpr int CT = Cfg<FP8, P>::kCT;     // tokens per chunk (one TMA box)
  if (FP8) {
    ok = make_tmap(&tmK, c.k_pool, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, kD, rows_tok, kD, CT,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    // V pages are d-major: rows of P token bytes; a chunk is a CT-byte column
    // band of the page's 128 rows
    const CUtensorMapSwizzle vsw = CT >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : CT == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                                 : CT == 32  ? CU_TENSOR_MAP_SWIZZLE_32B
                                             : CU_TENSOR_MAP_SWIZZLE_NONE;
    ok = ok && make_tmap(&tmV, c.v_pool, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, P,
                         (uint64_t)d.Lyr * d.S * d.Hkv * kD, CT, kD, vsw);
  } else {
    ok = make_tmap(&tmK, c.k_pool, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, rows_tok, 64, CT,
                   CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_tmap(&tmV, c.v_pool, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kD, rows_tok, 64, CT,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (!ok) return cudaErrorInvalidValue;
  const size_t smem = decode_smem<FP8, P>();
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<FP8, P>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int n = decode_grid<FP8, P>(d, a.n_layers, a.num_sms);
  if (n > decode_max_ctas(d, a.num_sms)) return cudaErrorInvalidValue;   // workspace bound
  p.w = d.max_selected();
  const long long T = (long long)a.n_layers * d.B * d.Hkv * p.w;
  if (T > INT_MAX / 2) return cudaErrorInvalidValue;
  p.T = (int)T;
  p.tq = p.T / n;
  p.tr = p.T % n;
  e = launch_pdl(decode_kernel<FP8, P>, dim3(n), dim3(kDecodeThreads), smem, s, p, tmK, tmV);
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
  p.Lp = d.Lp;
  p.nmax = d.nmax;
  p.bt = a.bt;
  p.slot_of = c.slot_of;
  p.k_mir = static_cast<const uint8_t*>(c.k_mirror);
  p.v_mir = static_cast<const uint8_t*>(c.v_mirror);
  p.ks_mir = c.k_scale_mirror;
  p.vs_mir = c.v_scale_mirror;
  switch (d.P * 2 + d.fp8) {
    case 32: return launch_decode_t<false, 16>(a, p, s);
    case 33: return launch_decode_t<true, 16>(a, p, s);
    case 64: return launch_decode_t<false, 32>(a, p, s);
    case 65: return launch_decode_t<true, 32>(a, p, s);
    case 128: return launch_decode_t<false, 64>(a, p, s);
    case 129: return launch_decode_t<true, 64>(a, p, s);
    case 256: return launch_decode_t<false, 128>(a, p, s);
    case 257: return launch_decode_t<true, 128>(a, p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssa
