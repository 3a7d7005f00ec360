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
//   * grid (split, b*Hkv+h, layer); each CTA takes a contiguous share of the
//     valid selected pages of its (layer, request, KV head);
//   * one producer warp streams each page's K and V (one KV head, P tokens)
//     into shared memory with TMA tiled copies (128-byte swizzle), plus the
//     fp8 per-token scales with bulk copies, through an mbarrier ring;
//   * four consumer warps each take 16-token blocks: QK^T and PV as
//     m16n8k16 tensor-core tiles with the G <= 8 query heads as the M rows,
//     fp32 accumulate, online softmax in the log2 domain with warp shuffles;
//   * bf16 K/V: bf16 MMAs, ldmatrix (V transposed by ldmatrix.trans);
//   * fp8 K/V: the e4m3 codes convert exactly to f16, so the MMAs run in f16
//     on the raw codes; q is scaled by a power of two into f16 range, the K
//     scale multiplies the fp32 score, and the V scale folds into the
//     probabilities (relative to a running power-of-two reference, so the
//     f16 operand never overflows).  V is stored d-major in the pool
//     ([Hkv][D][P]) so that the 8-bit reads run along tokens, the reduction
//     axis of PV;
//   * the 4 warps' states merge in shared memory; with several splits the
//     CTA writes (m, l, o) partials and a merge kernel combines them.
// The work is HBM-bound (8 flop/byte bf16, 16 fp8): the tensor cores carry
// the G-row tiles, the memory system sets the pace.
#include <cudaTypedefs.h>
#include <cuda.h>
#include <cmath>
#include <cstdio>

#include "common.cuh"
#include "internal.h"

namespace ssa {
namespace {

constexpr int kD = 128;
constexpr int kConsumerWarps = 4;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxG = 8;

__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

template <bool FP8, int P>
struct Cfg {
  static constexpr int kTileBytes = P * kD * (FP8 ? 1 : 2);      // one KV head of one page
  static constexpr int kScaleBytes = FP8 ? 2 * P * 4 : 0;
  static constexpr int kStageBytes = round_up(2 * kTileBytes + kScaleBytes, 1024);
  static constexpr int kStages = FP8 ? 4 : 3;
  static constexpr int kBlocks = P / 16;                          // 16-token blocks per page
  // log2 of the fp8 V^T row swizzle span in 16-byte units (row = P bytes)
  static constexpr int kVSwz = P >= 128 ? 3 : (P == 64 ? 2 : (P == 32 ? 1 : 0));
  static_assert(kConsumerWarps * kMaxG * kD * 4 + 2 * kConsumerWarps * kMaxG * 4 <=
                kStages * kStageBytes, "combine area must fit in the stage ring");
};

struct DecodeParams {
  const __nv_bfloat16* q;   // [n_layers][B][Hq][D]
  const int32_t* sel;       // [n_layers][B][W]
  const int32_t* phys;
  const int32_t* seq_lens;
  const float* k_scale;     // [Lyr][S][P]
  const float* v_scale;
  __nv_bfloat16* out;       // [n_layers][B][Hq][D]
  float* part_o;            // [units][splits][G][D]
  float* part_ml;           // [units][splits][G][2]
  int32_t* tickets;         // [units] split counters, zero between calls
  int32_t* status;
  int layer0, B, Hq, Hkv, G, W, S, splits;
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

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Producer warp -> consumer warps: the page list is written (barrier 2).
__device__ __forceinline__ void list_publish() {
  asm volatile("bar.arrive 2, %0;" ::"n"(kDecodeThreads) : "memory");
}
__device__ __forceinline__ void list_wait() {
  asm volatile("bar.sync 2, %0;" ::"n"(kDecodeThreads) : "memory");
}

// 1/x for x a positive normal power of two, exactly, without a division.
__device__ __forceinline__ float pow2_rcp(float x) {
  return __uint_as_float(0x7F000000u - __float_as_uint(x));
}

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

template <bool FP8, int P>
__global__ void __launch_bounds__(kDecodeThreads, FP8 ? 3 : 2)
decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV) {
  using C = Cfg<FP8, P>;
  constexpr int NST = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  int2* plist = reinterpret_cast<int2*>(smem + NST * C::kStageBytes);     // [W]
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(plist + round_up(p.W, 2));  // [8][D]
  uint64_t* full = reinterpret_cast<uint64_t*>(qs + kMaxG * kD);
  uint64_t* empty = full + NST;
  __shared__ int s_nv;
  __shared__ int s_abort;
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, bh = blockIdx.y, li = blockIdx.z;
  const int b = bh / p.Hkv, h = bh - b * p.Hkv;
  const int layer = p.layer0 + li;

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();                 // sel, phys, q and the pool come from earlier kernels
  const int seq_len = p.seq_lens[b];

  if (warp == kConsumerWarps) {
    // ---------------- producer warp: the page list, then one elected thread
    // issues every copy (the consumers meanwhile stage q) ----------------
    if (lane == 0) {
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
    }
    const int32_t* selr = p.sel + ((size_t)li * p.B + b) * p.W;
    const int32_t* physr = p.phys + ((size_t)li * p.B + b) * p.W;
    int cnt = 0;
    for (int base = 0; base < p.W; base += 32) {
      const int i = base + lane;
      int pg = -1, sl = -1;
      if (i < p.W) { pg = selr[i]; sl = physr[i]; }
      const bool ok = pg >= 0 && sl >= 0 && sl < p.S;
      if (pg >= 0 && sl < 0) set_status(p.status, SSA_ST_UNRESOLVED);
      if (pg >= 0 && sl >= p.S) set_status(p.status, SSA_ST_BAD_ID);
      const unsigned m = __ballot_sync(0xffffffffu, ok);
      if (ok) plist[cnt + __popc(m & ((1u << lane) - 1u))] = make_int2(pg, sl);
      cnt += __popc(m);
    }
    if (lane == 0) s_nv = cnt;
    list_publish();           // page list and count visible to the consumers
    const int i0 = (int)((long long)cnt * split / p.splits);
    const int nst = (int)((long long)cnt * (split + 1) / p.splits) - i0;
    if (lane != 0 || nst <= 0) return;
    int issued = 0;
    bool aborted = false;
    for (int st = 0; st < nst; ++st) {
      const int sb = st % NST;
      if (st >= NST && !mbar_wait(&empty[sb], ((st / NST) - 1) & 1, &s_abort)) {
        aborted = true;
        break;
      }
      const int2 e = plist[i0 + st];
      const int row_k = ((layer * p.S + e.y) * p.Hkv + h) * P;
      uint8_t* stage = ring + sb * C::kStageBytes;
      mbar_arrive_expect_tx(&full[sb], 2 * C::kTileBytes + C::kScaleBytes);
      if (FP8) {
        tma_load_2d(stage, &tmK, &full[sb], 0, row_k);
        const int row_v = ((layer * p.S + e.y) * p.Hkv + h) * kD;
        tma_load_2d(stage + C::kTileBytes, &tmV, &full[sb], 0, row_v);
        const size_t so = ((size_t)layer * p.S + e.y) * P;
        bulk_load(stage + 2 * C::kTileBytes, p.k_scale + so, P * 4, &full[sb]);
        bulk_load(stage + 2 * C::kTileBytes + P * 4, p.v_scale + so, P * 4, &full[sb]);
      } else {
        tma_load_2d(stage, &tmK, &full[sb], 0, row_k);
        tma_load_2d(stage + P * 128, &tmK, &full[sb], 64, row_k);
        tma_load_2d(stage + C::kTileBytes, &tmV, &full[sb], 0, row_k);
        tma_load_2d(stage + C::kTileBytes + P * 128, &tmV, &full[sb], 64, row_k);
      }
      ++issued;
    }
    if (aborted) {
      s_abort = 1;
      set_status(p.status, SSA_ST_TIMEOUT);
      // let every copy still in flight land before the CTA can exit
      for (int st = issued > NST ? issued - NST : 0; st < issued; ++st)
        mbar_wait(&full[st % NST], (st / NST) & 1, nullptr);
    }
    return;
  }

  // the G query rows of this KV head (rows >= G are zero)
  {
    const uint4* src = reinterpret_cast<const uint4*>(
        p.q + (((size_t)li * p.B + b) * p.Hq + (size_t)h * p.G) * kD);
    uint4* dst = reinterpret_cast<uint4*>(qs);
    for (int i = tid; i < kMaxG * kD / 8; i += kConsumerWarps * 32) {
      const int g = i / (kD / 8);
      dst[i] = g < p.G ? src[i] : make_uint4(0, 0, 0, 0);
    }
  }
  consumer_sync();

  // ---------------- consumers -------------------------------------------------
  // QK^T: A = 16 K rows (tokens), B = q^T (8 heads), C = S^T[token][head].
  // PV:   A = V^T rows (16 of d), B = P^T (C transposed in registers by
  //       movmatrix), C = O^T[d][head].  No MMA row is padding.
  const int r4 = lane >> 2, c = lane & 3;

  // q^T as the B operand: b0 = q[r4][k 2c, 2c+1], b1 = q[r4][k 2c+8, 2c+9];
  // fp8: logical k pairs map to 4 consecutive bytes of K (d = 16ks+4c..+3)
  uint32_t qb[8][2];
  float qscale_log2 = p.sm_log2;
  if (FP8) {
    float amax = 0.0f;
    for (int i = lane; i < kMaxG * kD; i += 32) amax = fmaxf(amax, fabsf(__bfloat162float(qs[i])));
    amax = warp_max(amax);
    int eq = 0;
    if (amax > 0.0f) {
      const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFF);     // amax in [2^(ef-127), 2^(ef-126))
      eq = 141 - ef;                                                  // amax * 2^eq < 2^15
      eq = eq > 126 ? 126 : (eq < -126 ? -126 : eq);
    }
    const float up = exp2f((float)eq);
    qscale_log2 = p.sm_log2 * exp2f((float)-eq);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const __nv_bfloat16* r = qs + r4 * kD + 16 * ks + 4 * c;
      qb[ks][0] = pack_f16(__bfloat162float(r[0]) * up, __bfloat162float(r[1]) * up);
      qb[ks][1] = pack_f16(__bfloat162float(r[2]) * up, __bfloat162float(r[3]) * up);
    }
  } else {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qb[ks][0] = *reinterpret_cast<const uint32_t*>(qs + r4 * kD + 16 * ks + 2 * c);
      qb[ks][1] = *reinterpret_cast<const uint32_t*>(qs + r4 * kD + 16 * ks + 2 * c + 8);
    }
  }

  list_wait();              // the producer's page list
  const int nv = s_nv;
  const int i0 = (int)((long long)nv * split / p.splits);
  const int nst = (int)((long long)nv * (split + 1) / p.splits) - i0;

  float o[8][4];   // O^T: rows d = 16*mt + r4 (+8), columns (heads) 2c, 2c+1
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
  // softmax state of heads 2c, 2c+1 (the lanes that own those O^T columns);
  // fp8: probabilities carry v_scale / vref, vref a power of two above every
  // V scale seen so far (0 before the first block)
  float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.0f, l_run1 = 0.0f;
  float vref = FP8 ? 0.0f : 1.0f;
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

  for (int st = 0; st < nst; ++st) {
    const int sb = st % NST;
    if (!mbar_wait(&full[sb], (st / NST) & 1, &s_abort)) {
      s_abort = 1;
      set_status(p.status, SSA_ST_TIMEOUT);
      break;
    }
    const int2 e = plist[i0 + st];
    const int nvalid = max(0, min(P, seq_len - e.x * P));
    uint8_t* stage = ring + sb * C::kStageBytes;
    const uint32_t kb = smem_u32(stage);
    const uint32_t vb = kb + C::kTileBytes;
    const float* ksc = reinterpret_cast<const float*>(stage + 2 * C::kTileBytes);
    const float* vsc = ksc + P;

#pragma unroll 1
    for (int blk = 0; blk < C::kBlocks; ++blk) {
      if (((st * C::kBlocks + blk) & (kConsumerWarps - 1)) != warp) continue;
      const int tb = blk * 16;
      // zero V of the tokens past seq_len (their bytes are not ours to trust)
      if (nvalid < tb + 16) {
        if (FP8) {
          for (int i = lane; i < kD * 16; i += 32) {
            const int d = i >> 4, x = tb + (i & 15);
            if (x >= nvalid) stage[C::kTileBytes + swz(d * P + x, C::kVSwz)] = 0;
          }
        } else {
          for (int i = lane; i < 16 * 16; i += 32) {
            const int r = tb + (i >> 4), ch = i & 15;
            if (r >= nvalid)
              *reinterpret_cast<uint4*>(stage + C::kTileBytes + (ch >> 3) * (P * 128) + r * 128 +
                                        (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }

      // S^T = K q^T for 16 tokens; even and odd k-steps in two MMA chains
      float s[4] = {0.f, 0.f, 0.f, 0.f}, sx[4] = {0.f, 0.f, 0.f, 0.f};
      const int tkA = tb + tauA, tkB = tb + tauB;
      if (FP8) {
        const uint32_t rA = kb + tkA * 128 + 4 * c, rB = kb + tkB * 128 + 4 * c;
        const int xA = tkA & 7, xB = tkB & 7;
#pragma unroll
        for (int ks = 0; ks < 8; ks += 2) {
          const uint32_t wA0 = lds32(rA + ((ks ^ xA) << 4));
          const uint32_t wB0 = lds32(rB + ((ks ^ xB) << 4));
          const uint32_t wA1 = lds32(rA + (((ks + 1) ^ xA) << 4));
          const uint32_t wB1 = lds32(rB + (((ks + 1) ^ xB) << 4));
          uint32_t a0, a1, a2, a3, a4, a5, a6, a7;
          e4m3x4_to_f16x2x2(wA0, a0, a2);
          e4m3x4_to_f16x2x2(wB0, a1, a3);
          e4m3x4_to_f16x2x2(wA1, a4, a6);
          e4m3x4_to_f16x2x2(wB1, a5, a7);
          mma_f16(s, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
          mma_f16(sx, a4, a5, a6, a7, qb[ks + 1][0], qb[ks + 1][1]);
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
          mma_bf16(s, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
          mma_bf16(sx, a4, a5, a6, a7, qb[ks + 1][0], qb[ks + 1][1]);
        }
      }
      // rows: s[0], s[1] = token tkA, heads 2c, 2c+1; s[2], s[3] = token tkB
      float x0 = (s[0] + sx[0]) * qscale_log2, x1 = (s[1] + sx[1]) * qscale_log2;
      float x2 = (s[2] + sx[2]) * qscale_log2, x3 = (s[3] + sx[3]) * qscale_log2;
      float vsA = 0.0f, vsB = 0.0f;
      if (FP8) {
        const float kA = ksc[tkA], kB = ksc[tkB];
        x0 *= kA; x1 *= kA; x2 *= kB; x3 *= kB;
        vsA = vsc[tkA];
        vsB = vsc[tkB];
      }
      if (nvalid < tb + 16) {          // the tail of a request's last page
        if (tkA >= nvalid) { x0 = x1 = -INFINITY; vsA = 0.0f; }
        if (tkB >= nvalid) { x2 = x3 = -INFINITY; vsB = 0.0f; }
      }
      // per-head maxima over the 16 tokens: the 8 lanes r4 = 0..7 of this c
      float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
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
      const float p0 = fast_exp2(x0 - mu0), p1 = fast_exp2(x1 - mu1);
      const float p2 = fast_exp2(x2 - mu0), p3 = fast_exp2(x3 - mu1);
      uint32_t P0, P1;
      if (FP8) {
        l_run0 = l_run0 * corr0 + (p0 + p2);
        l_run1 = l_run1 * corr1 + (p1 + p3);
        const float wA = vsA * vinv, wB = vsB * vinv;
        P0 = pack_f16(p0 * wA, p1 * wA);
        P1 = pack_f16(p2 * wB, p3 * wB);
      } else {
        const float q0 = bf16_round(p0), q1 = bf16_round(p1);
        const float q2 = bf16_round(p2), q3 = bf16_round(p3);
        l_run0 = l_run0 * corr0 + (q0 + q2);
        l_run1 = l_run1 * corr1 + (q1 + q3);
        P0 = pack_bf16(q0, q1);
        P1 = pack_bf16(q2, q3);
      }
      m_run0 = mn0;
      m_run1 = mn1;
      if (__any_sync(0xffffffffu, oc0 != 1.0f || oc1 != 1.0f)) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][0] *= oc0; o[mt][1] *= oc1; o[mt][2] *= oc0; o[mt][3] *= oc1;
        }
      }
      // P^T as the B operand: each 8x8 half transposed across the warp
      const uint32_t b0 = movmatrix_trans(P0), b1 = movmatrix_trans(P1);

      // O^T += V^T P^T, 16 rows of d per MMA
      if (FP8) {
        // rows d = 16*mt + r4 and +8: the swizzle bits do not depend on mt
        // (16*P*mt is a multiple of the swizzle period), so hoist them
        const uint32_t va0 = vb + swz(r4 * P + tb + 4 * c, C::kVSwz);
        const uint32_t va1 = vb + swz((r4 + 8) * P + tb + 4 * c, C::kVSwz);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t w0 = lds32(va0 + mt * 16 * P);
          uint32_t w1 = lds32(va1 + mt * 16 * P);
          w0 = __funnelshift_l(w0, w0, rot);
          w1 = __funnelshift_l(w1, w1, rot);
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2x2(w0, a0, a2);
          e4m3x4_to_f16x2x2(w1, a1, a3);
          mma_f16(o[mt], a0, a1, a2, a3, b0, b1);
        }
      } else {
        const int mi = lane >> 3, rr = lane & 7;
        const int t = tb + (mi >> 1) * 8 + rr;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int chunk = 2 * mt + (mi & 1);
          const uint32_t addr =
              vb + (chunk >> 3) * (P * 128) + t * 128 + (((chunk & 7) ^ (t & 7)) << 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(a0, a1, a2, a3, addr);
          mma_bf16(o[mt], a0, a1, a2, a3, b0, b1);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[sb]);
  }

  // ---------------- merge the 4 warps' states (stage ring is idle now) ------
  // l: sum over the 8 lanes (r4) that share heads 2c, 2c+1
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l_run0 += __shfl_xor_sync(0xffffffffu, l_run0, off);
    l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, off);
  }
  consumer_sync();
  float* cO = reinterpret_cast<float*>(ring);                  // [4][8][D]
  float* cM = cO + kConsumerWarps * kMaxG * kD;                 // [4][8]
  float* cL = cM + kConsumerWarps * kMaxG;                      // [4][8]
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int d = 16 * mt + r4;
    cO[(warp * kMaxG + 2 * c) * kD + d] = o[mt][0] * vref;
    cO[(warp * kMaxG + 2 * c + 1) * kD + d] = o[mt][1] * vref;
    cO[(warp * kMaxG + 2 * c) * kD + d + 8] = o[mt][2] * vref;
    cO[(warp * kMaxG + 2 * c + 1) * kD + d + 8] = o[mt][3] * vref;
  }
  if (r4 == 0) {
    cM[warp * kMaxG + 2 * c] = m_run0;
    cM[warp * kMaxG + 2 * c + 1] = m_run1;
    cL[warp * kMaxG + 2 * c] = l_run0;
    cL[warp * kMaxG + 2 * c + 1] = l_run1;
  }
  consumer_sync();
  const int unit = (li * p.B + b) * p.Hkv + h;
  for (int i = tid; i < kMaxG * kD; i += kConsumerWarps * 32) {
    const int gg = i / kD, d = i - gg * kD;
    if (gg >= p.G) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cM[w * kMaxG + gg]);
    float L = 0.0f, O = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float f = fast_exp2(cM[w * kMaxG + gg] - M);
        L += cL[w * kMaxG + gg] * f;
        O += cO[(w * kMaxG + gg) * kD + d] * f;
      }
    }
    if (p.splits == 1) {
      const float r = L > 0.0f ? O / L : 0.0f;
      p.out[(((size_t)li * p.B + b) * p.Hq + h * p.G + gg) * kD + d] = __float2bfloat16_rn(r);
    } else {
      const size_t pi = ((size_t)unit * p.splits + split) * p.G + gg;
      p.part_o[pi * kD + d] = O;
      if (d == 0) {
        p.part_ml[pi * 2] = M;
        p.part_ml[pi * 2 + 1] = L;
      }
    }
  }
  if (p.splits == 1) return;

  // ---------------- a7: the last CTA of this unit merges the splits ---------
  // (an atomic ticket; no CTA ever waits for another)
  __threadfence();
  consumer_sync();
  if (tid == 0) s_last = atomicAdd(&p.tickets[unit], 1) == p.splits - 1;
  consumer_sync();
  if (!s_last) return;
  __threadfence();
  // one pass: per head, the splits' weights exp2(m_s - M) and 1/L in shared
  // memory (the ring is idle), then every output sums its splits' partials
  float* sF = reinterpret_cast<float*>(ring);              // [splits][8]
  float* sInvL = sF + p.splits * kMaxG;                     // [8]
  const size_t ub = (size_t)unit * p.splits * p.G;
  if (tid < p.G) {
    float M = -INFINITY;
    for (int sp = 0; sp < p.splits; ++sp)
      M = fmaxf(M, __ldcg(&p.part_ml[(ub + (size_t)sp * p.G + tid) * 2]));
    float L = 0.0f;
    for (int sp = 0; sp < p.splits; ++sp) {
      const size_t pi = ub + (size_t)sp * p.G + tid;
      const float f = M == -INFINITY ? 0.0f : fast_exp2(__ldcg(&p.part_ml[pi * 2]) - M);
      sF[sp * kMaxG + tid] = f;
      L += __ldcg(&p.part_ml[pi * 2 + 1]) * f;
    }
    sInvL[tid] = L > 0.0f ? 1.0f / L : 0.0f;
  }
  consumer_sync();
  for (int i = tid; i < p.G * kD; i += kConsumerWarps * 32) {
    const int gg = i / kD, d = i - gg * kD;
    float O = 0.0f;
#pragma unroll 4
    for (int sp = 0; sp < p.splits; ++sp)
      O += sF[sp * kMaxG + gg] * __ldcg(&p.part_o[(ub + (size_t)sp * p.G + gg) * kD + d]);
    p.out[(((size_t)li * p.B + b) * p.Hq + h * p.G + gg) * kD + d] =
        __float2bfloat16_rn(O * sInvL[gg]);
  }
  if (tid == 0) p.tickets[unit] = 0;     // ready for the next call
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
size_t decode_smem(int W) {
  using C = Cfg<FP8, P>;
  return 1024 + (size_t)C::kStages * C::kStageBytes + (size_t)round_up(W, 2) * 8 +
         kMaxG * kD * 2 + 2 * C::kStages * 8;
}

template <bool FP8, int P>
cudaError_t launch_decode_t(const DecodeArgs& a, const DecodeParams& p, cudaStream_t s) {
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
  const size_t smem = decode_smem<FP8, P>(d.W);
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<FP8, P>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.splits, d.B * d.Hkv, a.n_layers);
  e = launch_pdl(decode_kernel<FP8, P>, grid, dim3(kDecodeThreads), smem, s, p, tmK, tmV);
  count_launch();
  return e;
}

}  // namespace

// Resident CTAs per SM: the register cap of the launch bounds, or the
// shared-memory footprint, whichever is tighter.
int decode_ctas_per_sm(const Dims& d) {
  size_t smem;
  switch (d.P * 2 + d.fp8) {
    case 32: smem = decode_smem<false, 16>(d.W); break;
    case 33: smem = decode_smem<true, 16>(d.W); break;
    case 64: smem = decode_smem<false, 32>(d.W); break;
    case 65: smem = decode_smem<true, 32>(d.W); break;
    case 128: smem = decode_smem<false, 64>(d.W); break;
    case 129: smem = decode_smem<true, 64>(d.W); break;
    case 256: smem = decode_smem<false, 128>(d.W); break;
    default: smem = decode_smem<true, 128>(d.W); break;
  }
  const int by_regs = d.fp8 ? 3 : 2;
  const int by_smem = (int)((228u * 1024u) / (smem + 1024u));
  return by_smem < 1 ? 1 : (by_smem < by_regs ? by_smem : by_regs);
}

// Splits of each (layer, request, KV head) unit: as many as fill ONE wave of
// resident CTAs (a partial second wave would double the tail), at least two
// pages per split.
int decode_splits(const Dims& d, int n_layers, int num_sms) {
  const long long units = (long long)n_layers * d.B * d.Hkv;
  const long long slots = (long long)num_sms * decode_ctas_per_sm(d);
  long long s = slots / units;
  const int max_s = d.max_selected() / 2 > 1 ? d.max_selected() / 2 : 1;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  return (int)s;
}

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
  p.splits = a.splits;
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
