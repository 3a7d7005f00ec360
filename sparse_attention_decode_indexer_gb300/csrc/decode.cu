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
//     of a piece, valid tokens, unit, q slot).  Per unit the producer also
//     writes the unit's G query rows, loaded one unit ahead, as the QK B
//     operand into one of two q slots.  Empty pieces and the end of the range
//     travel as stages without data;
//   * QK^T on the 5th-generation tensor cores: one thread issues, per page,
//     tcgen05 MMAs with M = 64 (A = the page's K rows straight from the TMA
//     tile, tokens as rows), N = 16 (B = the q slot), accumulating S^T in
//     TMEM (16 columns per stage), and commits them to the stage's barrier;
//   * four consumer warps each take 16-token blocks: a warp reads its
//     block's 16 TMEM lanes as the m16n8 fragment, runs the online softmax in
//     the log2 domain with warp shuffles, and PV with d as the rows (A = V^T,
//     B = P^T, the probabilities transposed in registers by movmatrix) in
//     warp-level m16n8k16 MMAs, fp32 accumulate;
//   * bf16 K/V: bf16 MMAs (kind::f16 for QK), V by ldmatrix.trans;
//   * fp8 K/V: QK runs as kind::f8f6f4 e4m3 MMAs on the raw K codes, q scaled
//     by a power of two and split into two e4m3 terms (hi, lo: the B rows 0-7
//     and 8-15); the K scale multiplies the fp32 score.  The e4m3 V codes
//     convert exactly to f16 for PV, and the V scale folds into the
//     probabilities (relative to a running power-of-two reference, so the f16
//     operand never overflows).  V is stored d-major in the pool
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
#include <algorithm>
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
constexpr int kMmaWarp = kConsumerWarps + 2;
constexpr int kDecodeThreads = kConsumers + 96;
constexpr int kMaxG = 8;
constexpr int kWindow = 32;          // producer compaction window (entries)
constexpr int kMaxStages = 12;
constexpr int kSmemPerSm = 228 * 1024;
constexpr int kSmemPerCtaMax = 227 * 1024;
constexpr int kSmemReservedPerCta = 1024;

// stage descriptor flags
constexpr int kFirst = 1;   // first page of a piece: the stage also holds q
constexpr int kLast = 2;    // last page of a piece: flush after it
constexpr int kEmpty = 4;   // a piece without pages (no data in the stage)
constexpr int kDone = 8;    // end of the CTA's range
constexpr int kFinal = 16;  // with kLast / kEmpty: the CTA's last piece

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

template <bool FP8, int P>
struct Cfg {
  static constexpr int kTileBytes = P * kD * (FP8 ? 1 : 2);      // one KV head of one page
  static constexpr int kScaleBytes = FP8 ? 2 * P * 4 : 0;
  static constexpr int kStageBytes = round_up(2 * kTileBytes + kScaleBytes, 1024);
  static constexpr int kCombineBytes =
      round_up(kConsumerWarps * kMaxG * kD * 4 + 2 * kConsumerWarps * kMaxG * 4, 1024);
  // the QK B operand of a unit: 16 rows (N) of q, K-major, 128-byte swizzle;
  // fp8 one 128-byte slab (rows 0-7 the hi codes, 8-15 the lo codes), bf16
  // two 64-column slabs (rows 8-15 zero).  Two slots: consecutive units.
  static constexpr int kQTileBytes = FP8 ? 16 * 128 : 2 * 16 * 128;
  // QK runs as M = 64 MMAs (P = 128: two, over the page's halves); below 64
  // tokens the A operand starts up to 48 rows before the page so that its
  // tokens land on the TMEM lanes of the warps that take them, and reads up
  // to 64 rows from there: the shared memory before the ring (combine area,
  // q slots) and kAOver bytes past the last stage must exist
  static constexpr int kHalves = P == 128 ? 2 : 1;
  static constexpr int kRowsBefore = P < 64 ? 64 - P : 0;
  static constexpr int kAOverRaw = (FP8 ? 64 * 128 : P * 128 + 64 * 128) - kStageBytes;
  static constexpr int kAOver = P < 64 && kAOverRaw > 0 ? kAOverRaw : 0;
  static constexpr int kNCols = 16;                               // D columns of one M = 64 MMA
  static constexpr int kDCols = kNCols * kHalves;                 // per stage
  // alignment slack, combine area, q slots, producer window, descriptors,
  // barriers, over-read pad
  static constexpr int kFixed = 1024 + kCombineBytes + 2 * kQTileBytes + kWindow * 8 +
                                kMaxStages * 40 + 64 + kAOver;
  // two CTAs per SM when at least two stages fit beside the second CTA
  static constexpr int kStages2 = (kSmemPerSm / 2 - kSmemReservedPerCta - kFixed) / kStageBytes;
  static constexpr int kCtasPerSm = kStages2 >= 2 ? 2 : 1;
  static constexpr int kStagesFit =
      kCtasPerSm == 2 ? kStages2 : (kSmemPerCtaMax - kFixed) / kStageBytes;
  static constexpr int kStages = kStagesFit > kMaxStages ? kMaxStages : kStagesFit;
  static constexpr int kBlocks = P / 16;                          // 16-token blocks per page
  // log2 of the fp8 V^T row swizzle span in 16-byte units (row = P bytes)
  static constexpr int kVSwz = P >= 128 ? 3 : (P == 64 ? 2 : (P == 32 ? 1 : 0));
  // TMEM columns: a power of two >= 32.  At most two CTAs of this kernel fit
  // on an SM (shared memory), so two allocations of <= 256 columns never
  // exceed the SM's 512 and an allocation never waits.
  static constexpr int kTmemCols = kStages * kDCols <= 32    ? 32
                                   : kStages * kDCols <= 64  ? 64
                                   : kStages * kDCols <= 128 ? 128
                                                             : 256;
  // layout from the 1024-aligned base: combine area, q slots, the stage ring,
  // producer window, stage descriptors, barriers (full, empty, sfull [NST];
  // cfull, cfree, cbar), then the over-read pad
  static constexpr int kOffQ = kCombineBytes;
  static constexpr int kOffRing = kOffQ + 2 * kQTileBytes;
  static constexpr int kOffPlist = kOffRing + kStages * kStageBytes;
  static constexpr int kOffMeta = kOffPlist + kWindow * 8;
  static constexpr int kOffBars = kOffMeta + kStages * 16;
  static constexpr int kSmemBytes = 1024 + kOffBars + (3 * kStages + 3) * 8 + kAOver;
  static_assert(kStages >= 2, "at least two stages");
  static_assert(kStages * kDCols <= 256, "TMEM: at most 256 columns per CTA");
  static_assert(3 * kSmemBytes > kSmemPerSm, "a third CTA on the SM would overrun TMEM");
  static_assert(kSmemBytes <= kSmemPerCtaMax, "shared memory");
  static_assert(kRowsBefore * 128 <= kCombineBytes + 2 * kQTileBytes, "A over-read before the ring");
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
  int k5d;                  // fp8 K map: 1 = one 5-D box per page, 0 = 3-D boxes of 8 rows
  float sm_log2;            // sm_scale * log2(e)
};

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

// 3-D and 5-D tiled TMA loads (the fp8 K pages: rows permuted within 16-token blocks)
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(smem_dst)), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_5d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      ::"r"(smem_u32(smem_dst)), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
        "r"(smem_u32(bar))
      : "memory");
}

// ---- 5th-generation tensor cores (tcgen05): TMEM, MMA, TMEM -> registers ----
// Allocation by one whole warp; the column base is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(dst)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout (rows of 128 bytes, 16-byte chunk j of row r at chunk
// j ^ (r & 7), groups of 8 rows 1024 bytes apart).  A K step inside the
// 128-byte row advances the start address; the swizzle is a function of the
// address bits, so the tile base must be 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)     // start address >> 4
         | (1ull << 16)                          // leading-dimension offset (unused when swizzled)
         | ((uint64_t)(1024 >> 4) << 32)         // stride between 8-row groups
         | (1ull << 46)                          // descriptor version
         | (2ull << 61);                         // 128-byte swizzle
}

// Instruction descriptor: D f32, A and B K-major, M = 64, N = 16;
// kind::f8f6f4 with e4m3 A and B, or kind::f16 with bf16 A and B.
template <bool FP8>
__device__ __forceinline__ constexpr uint32_t qk_idesc() {
  return (1u << 4)                               // D format f32
         | ((FP8 ? 0u : 1u) << 7)                // A: e4m3 / bf16
         | ((FP8 ? 0u : 1u) << 10)               // B: e4m3 / bf16
         | ((16u >> 3) << 17)                    // N >> 3
         | ((64u >> 4) << 24);                   // M >> 4
}

// D[tmem] (+)= A B^T, one thread issues
template <bool FP8>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
  if (FP8)
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n"
                 ::"r"(d), "l"(a), "l"(b), "r"(qk_idesc<FP8>()), "r"(acc) : "memory");
  else
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 ::"r"(d), "l"(a), "l"(b), "r"(qk_idesc<FP8>()), "r"(acc) : "memory");
}

// The mbarrier gets one arrival once every MMA this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}

// 16 TMEM lanes x 8 f32 columns -> the m16n8 accumulator fragment: lane
// (r4, c) gets (lane r4, columns 2c, 2c+1) and (lane r4 + 8, same columns).
// NT such loads at column offsets 0, 8, ..., then the wait; the registers
// pass through the wait so that no use can be scheduled before it.
template <int NT>
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[4 * NT]) {
  static_assert(NT == 1 || NT == 2, "one or two column groups");
  uint32_t r[4 * NT];
#pragma unroll
  for (int t = 0; t < NT; ++t)
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[4 * t]), "=r"(r[4 * t + 1]), "=r"(r[4 * t + 2]), "=r"(r[4 * t + 3])
                 : "r"(taddr + 8 * t) : "memory");
  if (NT == 1)
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]) :: "memory");
  else
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]),
                   "+r"(r[4 * NT - 4]), "+r"(r[4 * NT - 3]), "+r"(r[4 * NT - 2]), "+r"(r[4 * NT - 1])
                 :: "memory");
#pragma unroll
  for (int i = 0; i < 4 * NT; ++i) v[i] = __uint_as_float(r[i]);
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
  float* comb = reinterpret_cast<float*>(smem);
  uint8_t* qtile = smem + C::kOffQ;                                       // [2] q slots
  uint8_t* ring = smem + C::kOffRing;
  int2* plist = reinterpret_cast<int2*>(smem + C::kOffPlist);
  int4* meta = reinterpret_cast<int4*>(smem + C::kOffMeta);              // [NST]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* empty = full + NST;
  uint64_t* sfull = empty + NST;           // the stage's QK MMAs are done: S^T in TMEM
  uint64_t* cfull = sfull + NST;           // the consumers' states are in comb
  uint64_t* cfree = cfull + 1;             // the merge warp is done reading comb
  uint64_t* cbar = cfree + 1;              // the consumer warps' barrier (last piece)
  __shared__ int s_abort;
  __shared__ int s_last;
  __shared__ uint32_t s_tmem;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
      mbar_init(&sfull[i], 1);
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
  // TMEM for the scores: kDCols columns per stage (the MMA warp allocates
  // and frees it)
  if (warp == kMmaWarp) tmem_alloc(&s_tmem, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
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

  if (warp == kMmaWarp) {
    // ---------------- MMA warp -----------------------------------------------
    // Lane 0 issues the QK MMAs of each stage as soon as its data has landed,
    // in stage order, and commits them to the stage's sfull barrier; a stage
    // without data gets a plain arrival, so that sfull counts the ring's
    // phases and the consumers, who wait for it on every stage, never release
    // a stage this warp has not read.  A page below 64 tokens starts
    // 16 * ((pc * kBlocks) & 3) rows early so that its blocks land on the
    // TMEM lanes of the warps that take them (pc: data pages so far).
    const uint32_t tmem = s_tmem;
    if (lane == 0) {
      int pc = 0, n_st = 0;
      for (int st = 0;; ++st) {
        const int s2 = st % NST;
        if (!mbar_wait(&full[s2], (st / NST) & 1, &s_abort)) {
          s_abort = 1;
          set_status(p.status, SSA_ST_TIMEOUT);
          break;
        }
        const int4 d2 = meta[s2];
        if (d2.x & kDone) break;
        n_st = st + 1;
        if (d2.x & kEmpty) {
          mbar_arrive(&sfull[s2]);
          continue;
        }
        tc_fence_after();
        const int row0 = P < 64 ? 16 * ((pc * C::kBlocks) & 3) : 0;
        const uint32_t kt = smem_u32(ring + s2 * C::kStageBytes) - row0 * 128;
        const uint32_t qt = smem_u32(qtile + (d2.w & 1) * C::kQTileBytes);
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf) {
          const uint32_t dcol = tmem + s2 * C::kDCols + hf * C::kNCols;
#pragma unroll
          for (int ks = 0; ks < (FP8 ? 4 : 8); ++ks) {        // 32 bytes of K per MMA
            const int sl = FP8 ? 0 : ks >> 2;
            const uint32_t off = 32 * (ks & 3);
            const uint64_t ad = sw128_desc(kt + sl * P * 128 + hf * 64 * 128 + off);
            const uint64_t bd = sw128_desc(qt + sl * 2048 + off);
            tc_mma<FP8>(dcol, ad, bd, ks > 0);
          }
        }
        tc_commit(&sfull[s2]);
        ++pc;
      }
      // TMEM goes back only once every commit has arrived (the consumers
      // waited for each; after an abort this bounded wait covers the rest)
      for (int s3 = n_st > NST ? n_st - NST : 0; s3 < n_st; ++s3)
        mbar_wait(&sfull[s3 % NST], (s3 / NST) & 1, nullptr);
    }
    __syncwarp();
    tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers + 32) : "memory");   // consumers done with TMEM
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
    return;
  }

  if (warp == kProducerWarp) {
    // ---------------- producer warp ----------------------------------------
    // The warp reads and compacts the rows; lane 0 alone issues the copies.
    int st = 0;                 // stages issued (lane 0)
    bool ok = true;
    int cur_row = -1, cnt = 0, seq_len = 0;
    int pgc[4], slc[4];        // the row's first 128 entries, kept for the second pass

    auto acquire = [&](int s) -> bool {      // lane 0: stage slot s % NST is free
      return s < NST || mbar_wait(&empty[s % NST], ((s / NST) - 1) & 1, &s_abort);
    };
    auto issue_marker = [&](int kind, int unit) -> bool {   // lane 0
      if (!acquire(st)) return false;
      const int sb = st % NST;
      meta[sb] = make_int4(kind, 0, unit, 0);
      mbar_arrive(&full[sb]);
      ++st;
      return true;
    };

    // q of a unit -> the QK B operand (Cfg::kQTileBytes).  fp8: lane (g4 =
    // lane >> 3, j = lane & 7) takes d 16j..16j+15 of heads g4 and g4 + 4;
    // bf16: 16-byte chunk i = lane + 32k is slab i >> 6, head (i >> 3) & 7,
    // d 64 (i >> 6) + 8 (i & 7)..+7.  Heads >= G are zero.
    uint4 qraw[4];
    auto q_fetch = [&](int unit) {                        // all lanes
      const uint4* qg = reinterpret_cast<const uint4*>(p.q + (size_t)unit * p.G * kD);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        int g, off;                                       // head, 16-byte word in its row
        if (FP8) {
          g = (lane >> 3) + 4 * (k >> 1);
          off = 2 * (lane & 7) + (k & 1);
        } else {
          const int i = lane + 32 * k;
          g = (i >> 3) & 7;
          off = 8 * (i >> 6) + (i & 7);
        }
        qraw[k] = g < p.G ? qg[g * (kD / 8) + off] : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    // writes the tile of qraw into slot `slot`; returns the fp8 exponent eq
    // (q * 2^eq has its largest magnitude in [128, 256) and is split into two
    // e4m3 terms hi + lo, exact to 2^-10 of it, so QK runs on the raw K codes)
    auto q_build = [&](int slot) -> int {                 // all lanes
      uint8_t* qt = qtile + slot * C::kQTileBytes;
      int eq = 0;
      if (FP8) {
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) amax = fmaxf(amax, bf16x8_absmax(qraw[k]));
        amax = warp_max(amax);
        if (amax > 0.0f) {
          const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFF);  // amax in [2^(ef-127), 2^(ef-126))
          eq = 134 - ef;
          eq = eq > 126 ? 126 : (eq < -126 ? -126 : eq);
        }
        const float up = __uint_as_float((uint32_t)(eq + 127) << 23);
        const int j = lane & 7;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int g = (lane >> 3) + 4 * hh;
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint4 w = qraw[2 * hh + k];
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              const uint32_t a = ww[2 * m], b = ww[2 * m + 1];
              const float x0 = __uint_as_float(a << 16) * up, x1 = __uint_as_float(a & 0xFFFF0000u) * up;
              const float x2 = __uint_as_float(b << 16) * up, x3 = __uint_as_float(b & 0xFFFF0000u) * up;
              const uint32_t H = f32x4_to_e4m3x4(x0, x1, x2, x3);
              float y0, y1, y2, y3;
              e4m3x4_to_f32x4(H, y0, y1, y2, y3);
              hi[2 * k + m] = H;
              lo[2 * k + m] = f32x4_to_e4m3x4(x0 - y0, x1 - y1, x2 - y2, x3 - y3);
            }
          }
          *reinterpret_cast<uint4*>(qt + g * 128 + ((j ^ g) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(qt + (g + 8) * 128 + ((j ^ g) << 4)) =
              make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = lane + 32 * k, sl = i >> 6, g = (i >> 3) & 7, cc = i & 7;
          *reinterpret_cast<uint4*>(qt + sl * 2048 + g * 128 + ((cc ^ g) << 4)) = qraw[k];
          *reinterpret_cast<uint4*>(qt + sl * 2048 + (g + 8) * 128 + ((cc ^ g) << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // the tensor cores read the tile through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      return eq;
    };
    int n_built = 0;                  // q tiles built (slot = n_built & 1)
    int slot_last0 = -1, slot_last1 = -1;   // lane 0: last stage index that read each slot

    // lane 0: one page of K and V (one KV head) and its fp8 scales; qinfo =
    // q slot | (eq + 256) << 1
    auto issue_page = [&](int2 ent, int flags, int unit, int h, int layer, int seq_len,
                          int qinfo) -> bool {
      if (!acquire(st)) return false;
      const int sb = st % NST;
      const int nvalid = max(0, min(P, seq_len - ent.x * P));
      meta[sb] = make_int4(flags, nvalid, unit, qinfo);
      uint8_t* stage = ring + sb * C::kStageBytes;
      mbar_arrive_expect_tx(&full[sb], 2 * C::kTileBytes + C::kScaleBytes);
      const int row_k = ((layer * p.S + ent.y) * p.Hkv + h) * P;
      if (FP8) {
        if (p.k5d) {
          tma_load_5d(stage, &tmK, &full[sb], 0, 0, 0, 0, row_k / 16);
        } else {
#pragma unroll
          for (int blk = 0; blk < C::kBlocks; ++blk)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              tma_load_3d(stage + (16 * blk + 8 * hh) * 128, &tmK, &full[sb], 0, 2 * hh,
                          row_k / 4 + 4 * blk);
        }
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
      ++st;
      return true;
    };

    q_fetch(u_first);

    for (int u = u_first; u <= u_last && ok; ++u) {
      const int us = u * p.w;
      const int a = max(t0, us) - us;
      const int e = min(t1, us + p.w) - us;
      const int row = u / p.Hkv, h = u - row * p.Hkv;
      const int li = row / p.B, b = row - li * p.B;
      const int layer = p.layer0 + li;
      const int32_t* selr = p.sel + (size_t)row * p.W;
      const int32_t* physr = p.phys + (size_t)row * p.W;
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
            sl[k] = i < p.W ? physr[i] : -1;
            if (base == 0) { pgc[k] = pg[k]; slc[k] = sl[k]; }
          }
          int bad = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const bool valid = pg[k] >= 0 && sl[k] >= 0 && sl[k] < p.S;
            if (pg[k] >= 0 && sl[k] < 0) bad |= SSA_ST_UNRESOLVED;
            if (pg[k] >= 0 && sl[k] >= p.S) bad |= SSA_ST_BAD_ID;
            cnt += __popc(__ballot_sync(0xffffffffu, valid));
          }
          if (bad) set_status(p.status, bad);
        }
      }
      // this piece's share [a, e) of the unit's weight, as valid entries [j0, j1)
      const int j0 = (int)((long long)a * cnt / p.w), j1 = (int)((long long)e * cnt / p.w);
      if (j0 == j1) {
        if (u < u_last) q_fetch(u + 1);
        if (lane == 0) ok = issue_marker(kEmpty | (u == u_last ? kFinal : 0), u);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        continue;
      }
      // the q slot: the unit that used it before must be done with it, i.e.
      // the consumers released its last page (they wait for a page's MMAs
      // before they use it); the ring's own waits often show that already
      const int slot = n_built & 1;
      const int jl = slot ? slot_last1 : slot_last0;
      if (lane == 0 && jl >= 0 && st <= jl + NST)
        ok = mbar_wait(&empty[jl % NST], (jl / NST) & 1, &s_abort);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int eq = q_build(slot);
      const int qinfo = slot | ((eq + 256) << 1);
      ++n_built;
      if (u < u_last) q_fetch(u + 1);
      int seen = 0, issued = 0;
      for (int base = 0; base < p.W && seen < j1 && ok; base += 4 * 32) {
        int pgv[4], slv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = base + 32 * k + lane;
          pgv[k] = base == 0 ? pgc[k] : (i < p.W ? selr[i] : -1);
          slv[k] = base == 0 ? slc[k] : (i < p.W ? physr[i] : -1);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (seen >= j1 || !ok) break;
          const bool valid = pgv[k] >= 0 && slv[k] >= 0 && slv[k] < p.S;
          const unsigned lt = (1u << lane) - 1u;
          const unsigned m = __ballot_sync(0xffffffffu, valid);
          const int rank = seen + __popc(m & lt);
          const bool in = valid && rank >= j0 && rank < j1;
          const unsigned mi = __ballot_sync(0xffffffffu, in);
          if (in) plist[__popc(mi & lt)] = make_int2(pgv[k], slv[k]);
          __syncwarp();
          if (lane == 0) {
            const int nw = __popc(mi);
            for (int x = 0; x < nw && ok; ++x, ++issued) {
              const int flags = (issued == 0 ? kFirst : 0) |
                                (issued == j1 - j0 - 1 ? (u == u_last ? kLast | kFinal : kLast) : 0);
              ok = issue_page(plist[x], flags, u, h, layer, seq_len, qinfo);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          __syncwarp();                        // the window is rewritten next round
          seen += __popc(m);
        }
      }
      if (slot) slot_last1 = st - 1;
      else slot_last0 = st - 1;
    }
    if (lane != 0) return;
    if (ok) ok = issue_marker(kDone, 0);
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
  // QK^T: tcgen05 MMAs, M = 64 (A = the page's K rows, tokens), N = 16
  //       (B = the q tile), S^T[token][column] in TMEM; a warp reads the 16
  //       lanes of its 16-token block as the m16n8 fragment.
  // PV:   A = V^T rows (16 of d), B = P^T (S^T transposed in registers by
  //       movmatrix), C = O^T[d][head], warp-level MMAs.
  const int r4 = lane >> 2, c = lane & 3;
  const uint32_t tmem_w = s_tmem + ((uint32_t)(32 * warp) << 16);   // this warp's TMEM lanes

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
      if (dsc.x & kDone) break;
      // the MMA warp is through with the stage (data: S^T is in TMEM)
      if (!mbar_wait(&sfull[sb], (st / NST) & 1, &s_abort)) {
        s_abort = 1;
        set_status(p.status, SSA_ST_TIMEOUT);
        break;
      }
      tc_fence_after();
      if (dsc.x & kEmpty) {
        if (lane == 0) mbar_arrive(&empty[sb]);
        fkind = (dsc.x & kFinal) ? 2 : 1;
        funit = dsc.z;
        goto flushes;
      }
      const int nvalid = dsc.y;
      uint8_t* stage = ring + sb * C::kStageBytes;
      const uint32_t vb = smem_u32(stage) + C::kTileBytes;
      const float* ksc = reinterpret_cast<const float*>(stage + 2 * C::kTileBytes);
      const float* vsc = ksc + P;
      // fp8: the MMAs saw q * 2^eq
      if (FP8) qscale_log2 = p.sm_log2 * __uint_as_float((uint32_t)(127 - ((dsc.w >> 1) - 256)) << 23);

      constexpr int kSteps = C::kBlocks;
#pragma unroll 1
      for (int bs = 0; bs < kSteps; ++bs) {
        if (((pc * kSteps + bs) & (kConsumerWarps - 1)) != warp) continue;
        const int tb = bs * 16;
        // zero V of the tokens past seq_len (their bytes are not ours to trust)
        if (nvalid < tb + 16) {
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
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
        }
        // S^T of the block from TMEM: x[0], x[1] = token tkA, heads 2c, 2c+1;
        // x[2], x[3] = token tkB (fp8: the hi and lo columns summed).  fp8 K
        // rows arrive permuted (MMA row 8h + 2j + e = token 4j + 2h + e of the
        // block), so that MMA rows 2c, 2c+1, 2c+8, 2c+9 -- the k indices of
        // one lane's PV A operand -- are the 4 consecutive tokens 4c..4c+3.
        const int tkA = FP8 ? tb + 4 * (r4 >> 1) + (r4 & 1) : tb + r4;
        const int tkB = FP8 ? tkA + 2 : tb + r4 + 8;
        float x[4];
        {
          const uint32_t ta = tmem_w + sb * C::kDCols + (P == 128 ? (bs >> 2) * C::kNCols : 0);
          if (FP8) {
            float v[8];
            tmem_ld16<2>(ta, v);
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = (v[i] + v[4 + i]) * qscale_log2;
          } else {
            float v[4];
            tmem_ld16<1>(ta, v);
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = v[i] * qscale_log2;
          }
        }
        float vsA = 0.0f, vsB = 0.0f;
        if (FP8) {
          const float kA = ksc[tkA], kB = ksc[tkB];
          x[0] *= kA; x[1] *= kA; x[2] *= kB; x[3] *= kB;
          vsA = vsc[tkA];
          vsB = vsc[tkB];
        }
        if (nvalid < tb + 16) {            // the tail of a request's last page
          if (tkA >= nvalid) { x[0] = x[1] = -INFINITY; vsA = 0.0f; }
          if (tkB >= nvalid) { x[2] = x[3] = -INFINITY; vsB = 0.0f; }
        }
        // per-head maxima over the block's tokens: the 8 lanes r4 = 0..7 of c
        float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
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
          float vmax = fmaxf(vsA, vsB);
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
        uint32_t b0, b1;
        float ls0, ls1;
        {
          const float p0 = fast_exp2(x[0] - mu0), p1 = fast_exp2(x[1] - mu1);
          const float p2 = fast_exp2(x[2] - mu0), p3 = fast_exp2(x[3] - mu1);
          uint32_t P0, P1;
          if (FP8) {
            ls0 = p0 + p2;
            ls1 = p1 + p3;
            const float wA = vsA * vinv, wB = vsB * vinv;
            P0 = pack_f16(p0 * wA, p1 * wA);
            P1 = pack_f16(p2 * wB, p3 * wB);
          } else {
            const float q0 = bf16_round(p0), q1 = bf16_round(p1);
            const float q2 = bf16_round(p2), q3 = bf16_round(p3);
            ls0 = q0 + q2;
            ls1 = q1 + q3;
            P0 = pack_bf16(q0, q1);
            P1 = pack_bf16(q2, q3);
          }
          // P^T as the B operand: each 8x8 half transposed across the warp;
          // b0 = MMA rows 2c, 2c+1, b1 = rows 2c+8, 2c+9, head r4
          b0 = movmatrix_trans(P0);
          b1 = movmatrix_trans(P1);
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

        // O^T += V^T P^T, 16 rows of d per MMA
        if (FP8) {
          // A rows d = 16*mt + r4 and +8; k = 2c, 2c+1 (a0, a1) and 2c+8,
          // 2c+9 (a2, a3) are tokens 4c..4c+3: one 32-bit read of the d-major
          // V row.  The swizzle bits do not depend on mt (16*P*mt is a
          // multiple of the swizzle period), so hoist them.
          const uint32_t va0 = vb + swz(r4 * P + tb + 4 * c, C::kVSwz);
          const uint32_t va1 = vb + swz((r4 + 8) * P + tb + 4 * c, C::kVSwz);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            uint32_t a0, a1, a2, a3;
            e4m3x4_to_f16x2x2(lds32(va0 + mt * 16 * P), a0, a2);
            e4m3x4_to_f16x2x2(lds32(va1 + mt * 16 * P), a1, a3);
            mma_f16(o[mt], a0, a1, a2, a3, b0, b1);
          }
        } else {
          const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            const int t = tb + (mi >> 1) * 8 + rr;
            const int chunk = 2 * mt + (mi & 1);
            const uint32_t addr =
                vb + (chunk >> 3) * (P * 128) + t * 128 + (((chunk & 7) ^ (t & 7)) << 4);
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(a0, a1, a2, a3, addr);
            mma_bf16(o[mt], a0, a1, a2, a3, b0, b1);
          }
        }
      }
      tc_fence_before();
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

  // the MMA warp frees TMEM once the consumers are done reading it
  tc_fence_before();
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers + 32) : "memory");
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

// fp8 K pages with their rows permuted within each 16-token block: shared
// row 8h + 2j + e holds token 4j + 2h + e.  First choice, one box per page: a
// 5-D view (128 bytes, e: 2, j: 4, h: 2, 16-token blocks) with the byte
// strides 128, 512, 256, 2048.  If the driver will not encode that view, a
// 3-D view (128 bytes, 4 rows, groups of 4 rows) with boxes of (128, 2, 4)
// at row offset 2h: two boxes per block.
bool make_tmap_kperm(CUtensorMap* tm, void* base, uint64_t rows, int P, int* k5d) {
  auto fn = encode_fn();
  if (!fn) return false;
  {
    cuuint64_t dims[5] = {(cuuint64_t)kD, 2, 4, 2, rows / 16};
    cuuint64_t strides[4] = {128, 512, 256, 2048};
    cuuint32_t box[5] = {(cuuint32_t)kD, 2, 4, 2, (cuuint32_t)(P / 16)};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    if (fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, base, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      *k5d = 1;
      return true;
    }
  }
  cuuint64_t dims[3] = {(cuuint64_t)kD, 4, rows / 4};
  cuuint64_t strides[2] = {128, 512};
  cuuint32_t box[3] = {(cuuint32_t)kD, 2, 4};
  cuuint32_t estr[3] = {1, 1, 1};
  *k5d = 0;
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FP8, int P>
size_t decode_smem() {
  return (size_t)Cfg<FP8, P>::kSmemBytes;
}

// CTAs of one wave: resident CTAs per SM (the configuration's target, or
// what the kernel's registers and shared memory allow, whichever is lower)
// x SMs, cut so that every CTA gets at least two tiles and no unit more
// than 130 pieces.  (The runtime's occupancy calculator answers one CTA per
// SM for this TMEM-allocating kernel although two fit and run together; the
// TMEM budget is kept by construction, see Cfg::kTmemCols.)  No CTA waits
// for another, so a wave that does not fit only runs longer.
template <bool FP8, int P>
int decode_grid(const Dims& d, int n_layers, int num_sms) {
  static int occ = -1;
  if (occ < 0) {
    int o = Cfg<FP8, P>::kCtasPerSm, dev = 0, regs_sm = 65536, smem_sm = kSmemPerSm;
    cudaFuncAttributes fa{};
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaFuncGetAttributes(&fa, decode_kernel<FP8, P>) == cudaSuccess) {
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
      const int regs_cta = ((fa.numRegs * 32 + 255) / 256 * 256) * (kDecodeThreads / 32);
      const int smem_cta = (int)(decode_smem<FP8, P>() + fa.sharedSizeBytes) + kSmemReservedPerCta;
      const int by_regs = regs_cta > 0 ? regs_sm / regs_cta : o;
      const int by_smem = smem_cta > 0 ? smem_sm / smem_cta : o;
      o = std::min(o, std::min(by_regs, by_smem));
    } else {
      o = 1;
    }
    occ = o < 1 ? 1 : o;
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
  if (FP8) {
    ok = make_tmap_kperm(&tmK, c.k_pool, rows_tok, P, &p.k5d);
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
