// store.cu -- a0: store K/V through the write-through host mirror, update the
// indexer slab; and the residency-state reset.
//
// FreeToken PR #499, "Design": each stored token is also written to pinned
// host memory (over unified addressing), so evicting a slot never needs a
// write-back.  FreeToken PR #525 (mirror_store_quant): with fp8 the host copy
// receives the quantised e4m3 codes and their fp32 scales, so host copy and
// pool hold the same bytes.
//
// Work split: the tokens are cut into chunks (one token per chunk for short
// calls such as a decode-step append, one page's worth for long ones such as
// a prefill); a CTA handles every run of consecutive tokens of one logical
// page that starts in its chunk, run after run.  Within a run one thread per
// slab element accumulates the running sum in token order, so the result is
// independent of scheduling.  The run's input is read a batch of tokens at a
// time (every load of the batch in flight at once); K rows (and bf16 V rows)
// pass through shared memory so that the pool and the host mirror receive
// 16-byte stores; fp8 V of a full page is transposed in shared memory and
// written as 16-byte d-rows.  Rounding: IEEE fp32 division and rintf, e4m3
// round-to-nearest-even with saturation -- the same operations the
// definition states, one at a time.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace ssa {
namespace {

struct StoreParams {
  uint8_t *k_pool, *v_pool;
  float *k_scale, *v_scale;
  uint8_t *k_mir, *v_mir;
  float *k_scale_m, *v_scale_m;
  int8_t* slab;
  float* slab_scale;
  float* slab_sum;
  int32_t* slab_cnt;
  const int32_t* slot_of;
  const __nv_bfloat16 *k, *v;   // [n_layers][T][HD]
  const int64_t* pos;
  int T, chunk;
  int32_t* status;
  int layer0, Lp, S, Hkv, D, P, fp8;
};

constexpr int kMaxPage = 128;
constexpr int kTokBatch = 8;               // tokens whose loads are in flight together

__device__ __forceinline__ uint8_t e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// dynamic shared memory: [fp8: V of a full page, HD * P B][K rows of a token
// batch, kTokBatch * HD * esz B][bf16: V rows of the batch, the same]
__host__ __device__ inline size_t store_smem(int HD, int P, int fp8) {
  return fp8 ? (size_t)HD * P + (size_t)kTokBatch * HD : (size_t)2 * kTokBatch * HD * 2;
}

__global__ void __launch_bounds__(1024) store_kernel(StoreParams p) {
  extern __shared__ __align__(16) uint8_t dsm[];
  __shared__ float s_ks[kMaxPage], s_vs[kMaxPage];
  __shared__ int s_j[kMaxPage];
  __shared__ int s_start[kMaxPage];
  __shared__ int s_nstart, s_run;
  __shared__ float red[33];
  pdl_wait();
  const int li = blockIdx.y, layer = p.layer0 + li;
  const int tid = threadIdx.x, P = p.P, HD = p.Hkv * p.D;
  const int esz = p.fp8 ? 1 : 2;
  uint8_t* vt = dsm;                                            // fp8 only
  uint8_t* kst = dsm + (p.fp8 ? (size_t)HD * P : 0);
  uint8_t* vst = kst + (size_t)kTokBatch * HD * esz;            // bf16 only

  // the runs that start in this CTA's chunk, in token order (a chunk of one
  // token: thread 0 decides alone)
  const int c0 = blockIdx.x * p.chunk, nc = min(p.chunk, p.T - c0);
  if (tid < nc && (nc > 1 || tid == 0)) {
    const int t = c0 + tid;
    const int64_t x = p.pos[t];
    bool start = true;
    if (x < 0 || x / P >= p.Lp) {
      set_status(p.status, SSA_ST_BAD_ID);
      start = false;
    } else if (t > 0) {
      const int64_t prev = p.pos[t - 1];
      if (prev >= x) set_status(p.status, SSA_ST_BAD_POS);
      if (prev >= 0 && prev / P == x / P) start = false;      // inside a run
    }
    s_start[tid] = start ? t : -1;
  }
  if (nc > 1) __syncthreads();                    // nc is the same for the whole CTA
  if (tid == 0) {
    int n = 0;
    for (int i = 0; i < nc; ++i)
      if (s_start[i] >= 0) s_start[n++] = s_start[i];
    s_nstart = n;
  }
  __syncthreads();
  const int nstart = s_nstart;

  for (int ri = 0; ri < nstart; ++ri) {
    const int t0 = s_start[ri];
    const int64_t pos0 = p.pos[t0];
    const int pg = (int)(pos0 / P);
    // the page's slab running sum and its slot, loaded now so that their
    // latency overlaps the run-length scan; the sum stays in a register
    const size_t so = ((size_t)layer * p.Lp + pg) * HD;
    const int e = tid;                                         // this thread's slab element
    float sum = e < HD ? p.slab_sum[so + e] : 0.0f;
    int slot = p.slot_of[(size_t)layer * p.Lp + pg];
    // run length: consecutive tokens of the same page (at most P)
    if (tid == 0) s_run = P;
    __syncthreads();
    if (tid >= 1 && tid < P) {
      const int t = t0 + tid;
      bool ends = t >= p.T;
      if (!ends) {
        const int64_t x = p.pos[t];
        ends = x < 0 || x / P != pg;
        if (!ends && x <= p.pos[t - 1]) set_status(p.status, SSA_ST_BAD_POS);
      }
      if (ends) atomicMin(&s_run, tid);
    }
    __syncthreads();
    const int R = s_run;
    if (tid < R) s_j[tid] = (int)(p.pos[t0 + tid] % P);
    __syncthreads();

    if (slot >= p.S) {                                  // corrupt state: never write through it
      if (tid == 0) set_status(p.status, SSA_ST_BAD_ID);
      slot = -1;
    }
    const size_t pe = (size_t)HD * P;                  // elements per page block
    uint8_t* km = p.k_mir ? p.k_mir + ((size_t)layer * p.Lp + pg) * pe * esz : nullptr;
    uint8_t* vm = p.v_mir ? p.v_mir + ((size_t)layer * p.Lp + pg) * pe * esz : nullptr;
    uint8_t* kp = slot >= 0 ? p.k_pool + ((size_t)layer * p.S + slot) * pe * esz : nullptr;
    uint8_t* vp = slot >= 0 ? p.v_pool + ((size_t)layer * p.S + slot) * pe * esz : nullptr;
    const __nv_bfloat16* kin = p.k + ((size_t)li * p.T + t0) * HD;
    const __nv_bfloat16* vin = p.v + ((size_t)li * p.T + t0) * HD;

    // phase 1 (fp8): per-token scales, one warp per token
    if (p.fp8) {
      const int lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
      for (int r = warp; r < R; r += nw) {
        float ak = 0.0f, av = 0.0f;
        for (int x = lane; x < HD; x += 32) {
          ak = fmaxf(ak, fabsf(__bfloat162float(kin[(size_t)r * HD + x])));
          av = fmaxf(av, fabsf(__bfloat162float(vin[(size_t)r * HD + x])));
        }
        ak = warp_max(ak);
        av = warp_max(av);
        if (lane == 0) {
          const float sk = ak > 0.0f ? ak / 448.0f : 1.0f;
          const float sv = av > 0.0f ? av / 448.0f : 1.0f;
          s_ks[r] = sk;
          s_vs[r] = sv;
          const size_t so_m = ((size_t)layer * p.Lp + pg) * P + s_j[r];
          if (p.k_scale_m) { p.k_scale_m[so_m] = sk; p.v_scale_m[so_m] = sv; }
          if (slot >= 0) {
            const size_t so_p = ((size_t)layer * p.S + slot) * P + s_j[r];
            p.k_scale[so_p] = sk;
            p.v_scale[so_p] = sv;
          }
        }
      }
    }
    __syncthreads();

    // phase 2: codes and the slab running sum (token order), a batch of
    // tokens at a time; K rows (bf16: and V rows) leave through shared memory
    // as 16-byte stores (measured faster than byte stores from the registers,
    // one-token runs included)
    const bool full_page = (R == P);
    const int h = e / p.D, d = e - h * p.D;
    const int row16 = p.D * esz / 16;                  // 16-byte units per token row of a head
    for (int r0 = 0; r0 < R; r0 += kTokBatch) {
      const int nb = min(kTokBatch, R - r0);
      __nv_bfloat16 xk[kTokBatch], xv[kTokBatch];
#pragma unroll
      for (int i = 0; i < kTokBatch; ++i) {
        if (i < nb && e < HD) {
          xk[i] = kin[(size_t)(r0 + i) * HD + e];
          xv[i] = vin[(size_t)(r0 + i) * HD + e];
        }
      }
      if (e < HD) {
#pragma unroll
        for (int i = 0; i < kTokBatch; ++i) {
          if (i >= nb) break;
          const int r = r0 + i, j = s_j[r];
          if (p.fp8) {
            const uint8_t ck = e4m3(__bfloat162float(xk[i]) / s_ks[r]);
            const uint8_t cv = e4m3(__bfloat162float(xv[i]) / s_vs[r]);
            kst[(size_t)i * HD + e] = ck;
            if (full_page) {
              vt[(size_t)e * P + j] = cv;
            } else {
              const size_t offt = ((size_t)h * p.D + d) * P + j;   // V: [h][d][j]
              if (vm) vm[offt] = cv;
              if (vp) vp[offt] = cv;
            }
          } else {
            reinterpret_cast<__nv_bfloat16*>(kst)[(size_t)i * HD + e] = xk[i];
            reinterpret_cast<__nv_bfloat16*>(vst)[(size_t)i * HD + e] = xv[i];
          }
          sum = sum + __bfloat162float(xk[i]);
        }
      }
      __syncthreads();
      // token row (r, head hh): D * esz bytes at [hh][j][0..D) of the page
      const int nvec = nb * p.Hkv * row16;
      for (int q = tid; q < nvec; q += blockDim.x) {
        const int i = q / (p.Hkv * row16), rem = q - i * p.Hkv * row16;
        const int hh = rem / row16, c = rem - hh * row16;
        const size_t src = ((size_t)i * HD + (size_t)hh * p.D) * esz + (size_t)c * 16;
        const size_t off = ((size_t)hh * P + s_j[r0 + i]) * p.D * esz + (size_t)c * 16;
        const uint4 kv4 = *reinterpret_cast<const uint4*>(kst + src);
        if (km) *reinterpret_cast<uint4*>(km + off) = kv4;
        if (kp) *reinterpret_cast<uint4*>(kp + off) = kv4;
        if (!p.fp8) {
          const uint4 vv4 = *reinterpret_cast<const uint4*>(vst + src);
          if (vm) *reinterpret_cast<uint4*>(vm + off) = vv4;
          if (vp) *reinterpret_cast<uint4*>(vp + off) = vv4;
        }
      }
      __syncthreads();                                 // the staging rows are rewritten next
    }
    if (e < HD) p.slab_sum[so + e] = sum;

    // phase 3a (fp8, full page): V rows [h][d][0..P) out of shared memory, 16 B at a time
    if (p.fp8 && full_page) {
      const int vec_per_row = P / 16;
      for (int i = tid; i < HD * vec_per_row; i += blockDim.x) {
        const int x = i / vec_per_row, c = i - x * vec_per_row;
        const uint4 val = *reinterpret_cast<const uint4*>(vt + (size_t)x * P + c * 16);
        const size_t off = (size_t)x * P + c * 16;   // x = h*D + d
        if (vm) *reinterpret_cast<uint4*>(vm + off) = val;
        if (vp) *reinterpret_cast<uint4*>(vp + off) = val;
      }
    }

    // phase 3b: re-quantise the page's slab row
    const int cnt = p.slab_cnt[(size_t)layer * p.Lp + pg] + R;
    float amax = e < HD ? fabsf(sum / (float)cnt) : 0.0f;
    amax = block_max(amax, red);
    const float s = amax / 127.0f;
    if (e < HD) {
      const float mean = sum / (float)cnt;
      int c = 0;
      if (amax > 0.0f) c = (int)fminf(fmaxf(rintf(mean / s), -127.0f), 127.0f);
      p.slab[so + e] = (int8_t)c;
    }
    if (tid == 0) {
      p.slab_cnt[(size_t)layer * p.Lp + pg] = cnt;
      p.slab_scale[(size_t)layer * p.Lp + pg] = s;
    }
    __syncthreads();                                   // vt, s_j, s_run, red: the next run's
  }
}

__global__ void lru_init_kernel(int32_t* slot_of, int32_t* page_of, int32_t* last_use,
                                int32_t* clock, int Lyr, int Lp, int S, int identity) {
  pdl_wait();
  const size_t nL = (size_t)Lyr * Lp, nS = (size_t)Lyr * S;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nL; i += stride) {
    const int pgi = (int)(i % Lp);
    slot_of[i] = (identity && pgi < S) ? pgi : -1;
  }
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nS; i += stride) {
    const int s = (int)(i % S);
    page_of[i] = (identity && s < Lp) ? s : -1;
    last_use[i] = -1;
  }
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < (size_t)Lyr; i += stride)
    clock[i] = 0;
}

}  // namespace

cudaError_t launch_lru_init(const Dims& d, const ssa_cache& c, int identity, cudaStream_t s) {
  const size_t HD = (size_t)d.Hkv * d.D, n = (size_t)d.Lyr * d.Lp;
  cudaError_t e;
  if ((e = cudaMemsetAsync(c.slab, 0, n * HD, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(c.slab_sum, 0, n * HD * sizeof(float), s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(c.slab_scale, 0, n * sizeof(float), s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(c.slab_cnt, 0, n * sizeof(int32_t), s)) != cudaSuccess) return e;
  e = launch_pdl(lru_init_kernel, dim3(1024), dim3(256), 0, s, c.slot_of, c.page_of, c.last_use,
                 c.clock, d.Lyr, d.Lp, d.S, identity);
  count_launch();
  return e;
}

cudaError_t launch_store(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                         const void* k, const void* v, const int64_t* pos, int T,
                         int32_t* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  StoreParams p{};
  p.k_pool = static_cast<uint8_t*>(c.k_pool);
  p.v_pool = static_cast<uint8_t*>(c.v_pool);
  p.k_scale = c.k_scale;
  p.v_scale = c.v_scale;
  p.k_mir = static_cast<uint8_t*>(c.k_mirror);
  p.v_mir = static_cast<uint8_t*>(c.v_mirror);
  p.k_scale_m = c.k_scale_mirror;
  p.v_scale_m = c.v_scale_mirror;
  p.slab = c.slab;
  p.slab_scale = c.slab_scale;
  p.slab_sum = c.slab_sum;
  p.slab_cnt = c.slab_cnt;
  p.slot_of = c.slot_of;
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.pos = pos;
  p.T = T;
  p.status = status;
  p.layer0 = layer0;
  p.Lp = d.Lp; p.S = d.S; p.Hkv = d.Hkv; p.D = d.D; p.P = d.P; p.fp8 = d.fp8;
  if (d.Hkv * d.D > 1024 || d.P > kMaxPage) return cudaErrorInvalidValue;
  const int threads = d.Hkv * d.D;
  // a decode-step append stores one token per request: one CTA per token;
  // a prefill stores whole pages: one CTA per page-sized chunk of tokens
  p.chunk = T >= 4096 ? d.P : 1;
  const size_t smem = store_smem(d.Hkv * d.D, d.P, d.fp8);
  if (smem + 4096 > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(store_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  const unsigned nchunk = (unsigned)((T + p.chunk - 1) / p.chunk);
  cudaError_t e = launch_pdl(store_kernel, dim3(nchunk, n_layers), dim3(threads), smem, s, p);
  count_launch();
  return e;
}

}  // namespace ssa
