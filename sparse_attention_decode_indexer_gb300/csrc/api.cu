// api.cu -- the C ABI: argument checks, workspace layout, launches.
//
// Every entry point validates its arguments on the host, then only enqueues
// kernels on the caller's stream.  Nothing here synchronises, allocates or
// keeps a pointer past the call.
#include <climits>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace ssa {
namespace {

thread_local int g_last_cuda_error = 0;
thread_local long long g_launches = 0;

int fail_cuda(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return SSA_ERR_CUDA;
}

bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

// Validate the layout and fill the derived view.
int check_layout(const ssa_layout* lay, Dims& d) {
  if (!lay) return SSA_ERR_INVALID_ARG;
  d.P = lay->page_size; d.Hq = lay->n_q_heads; d.Hkv = lay->n_kv_heads; d.D = lay->head_dim;
  d.fp8 = lay->kv_dtype == SSA_KV_FP8_E4M3;
  d.Lyr = lay->n_layers; d.Lp = lay->logical_pages; d.S = lay->pool_slots;
  d.B = lay->batch; d.nmax = lay->max_pages; d.k = lay->block_topk; d.W = lay->max_sel;
  if (d.Lyr < 1 || d.Lp < 1 || d.S < 1 || d.B < 1 || d.nmax < 1 || d.k < 1 || d.Hq < 1 ||
      d.Hkv < 1)
    return SSA_ERR_INVALID_ARG;
  if (d.W != 2 * d.k + 8) return SSA_ERR_INVALID_ARG;
  if (lay->kv_dtype != SSA_KV_BF16 && lay->kv_dtype != SSA_KV_FP8_E4M3) return SSA_ERR_UNSUPPORTED;
  if (d.D != 128) return SSA_ERR_UNSUPPORTED;
  if (!(d.P == 16 || d.P == 32 || d.P == 64 || d.P == 128)) return SSA_ERR_UNSUPPORTED;
  if (d.Hq % d.Hkv != 0) return SSA_ERR_UNSUPPORTED;
  d.G = d.Hq / d.Hkv;
  if (d.G > 8) return SSA_ERR_UNSUPPORTED;
  if (!pow2(d.Hkv) || d.Hkv > 8) return SSA_ERR_UNSUPPORTED;
  // TMA coordinates are int32: every row index of the pool must fit
  const long long rows = (long long)d.Lyr * d.S * d.Hkv * (d.P > d.D ? d.P : d.D);
  if (rows >= INT_MAX) return SSA_ERR_UNSUPPORTED;
  if ((long long)d.B * d.W > 16384) return SSA_ERR_UNSUPPORTED;   // ensure sorts in shared memory
  if (d.nmax > 49152) return SSA_ERR_UNSUPPORTED;                  // select keeps scores in smem
  return SSA_OK;
}

int check_range(const Dims& d, int layer0, int n_layers) {
  if (layer0 < 0 || n_layers < 1 || layer0 + n_layers > d.Lyr) return SSA_ERR_INVALID_ARG;
  return SSA_OK;
}

bool has_mirror(const Dims& d, const ssa_cache* c) {
  if (d.fp8)
    return c->k_mirror && c->v_mirror && c->k_scale_mirror && c->v_scale_mirror;
  return c->k_mirror && c->v_mirror;
}

bool mirror_consistent(const Dims& d, const ssa_cache* c) {
  const bool any = c->k_mirror || c->v_mirror || c->k_scale_mirror || c->v_scale_mirror;
  return !any || has_mirror(d, c);
}

int check_cache(const Dims& d, const ssa_cache* c) {
  if (!c || !c->k_pool || !c->v_pool || !c->slab || !c->slot_of || !c->page_of || !c->last_use ||
      !c->clock)
    return SSA_ERR_INVALID_ARG;
  if (d.fp8 && (!c->k_scale || !c->v_scale)) return SSA_ERR_INVALID_ARG;
  if (!mirror_consistent(d, c)) return SSA_ERR_NO_MIRROR;
  return SSA_OK;
}

int num_sms() { return current_device_info().sms; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace: [scores | miss_page | miss_slot | n_miss | part_o | part_ml |
// tickets | idx_tickets], each sized for the whole layer range of the
// layout.  Only the tickets need a defined start (zero); every call leaves
// them zero.
struct WsLayout {
  size_t scores, miss_page, miss_slot, n_miss, part_o, part_ml, tickets, idx_tickets;
  size_t pf_cand, pf_ncand, pf_miss_page, pf_miss_slot, pf_n_miss;   // ssa_prefetch_pages
  size_t total;
};

size_t part_entries(const Dims& d) {
  return (size_t)decode_max_ctas(d, num_sms()) * 2 * d.G;
}

WsLayout ws_layout(const Dims& d) {
  WsLayout w{};
  size_t off = 0;
  w.scores = off;    off += align256((size_t)d.Lyr * d.B * d.nmax * 4);
  w.miss_page = off; off += align256((size_t)d.Lyr * d.B * d.W * 4);
  w.miss_slot = off; off += align256((size_t)d.Lyr * d.B * d.W * 4);
  w.n_miss = off;    off += align256((size_t)d.Lyr * 4);
  const size_t pe = part_entries(d);
  w.part_o = off;    off += align256(pe * d.D * 4);
  w.part_ml = off;   off += align256(pe * 2 * 4);
  w.tickets = off;   off += align256((size_t)d.Lyr * d.B * d.Hkv * 4);
  w.idx_tickets = off; off += align256((size_t)d.Lyr * d.B * 4);
  w.pf_cand = off;   off += align256((size_t)d.Lyr * d.B * d.W * 4);
  w.pf_ncand = off;  off += align256((size_t)d.Lyr * d.B * 4);
  w.pf_miss_page = off; off += align256((size_t)d.Lyr * d.B * d.W * 4);
  w.pf_miss_slot = off; off += align256((size_t)d.Lyr * d.B * d.W * 4);
  w.pf_n_miss = off; off += align256((size_t)d.Lyr * 4);
  w.total = off;
  return w;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace

void count_launch(int n) { g_launches += n; }

// One entry per device ordinal, filled on first use with that device current.
// A host may hold GPUs of different kinds, so nothing is shared between them.
DeviceInfo current_device_info() {
  static std::mutex mu;
  static DeviceInfo info[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return DeviceInfo{152, 227 * 1024};
  std::lock_guard<std::mutex> lock(mu);
  DeviceInfo& d = info[dev];
  if (d.sms == 0) {
    int sms = 0, smem = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms < 1)
      sms = 152;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        smem < 48 * 1024)
      smem = 48 * 1024;
    d.smem_optin = smem;
    d.sms = sms;
  }
  return d;
}

int current_device_ordinal() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return dev;
}

int validate_layout(const ssa_layout* lay, Dims& d) { return check_layout(lay, d); }

int record_cuda_error(cudaError_t e) { return fail_cuda(e); }

}  // namespace ssa

using namespace ssa;

extern "C" {

size_t ssa_workspace_size(const ssa_layout* lay) {
  Dims d;
  if (check_layout(lay, d) != SSA_OK) return 0;
  return ws_layout(d).total;
}

int ssa_lru_init(const ssa_layout* lay, const ssa_cache* c, int identity, ssa_stream_t stream) {
  Dims d;
  int r = check_layout(lay, d);
  if (r) return r;
  if ((r = check_cache(d, c))) return r;
  if (!c->slab_scale || !c->slab_sum || !c->slab_cnt) return SSA_ERR_INVALID_ARG;
  cudaError_t e = launch_lru_init(d, *c, identity ? 1 : 0, (cudaStream_t)stream);
  return e == cudaSuccess ? SSA_OK : fail_cuda(e);
}

int ssa_store_kv_mirror(const ssa_layout* lay, const ssa_cache* c, int layer0, int n_layers,
                        const void* k, const void* v, const int64_t* pos, int T,
                        int32_t* status, ssa_stream_t stream) {
  Dims d;
  int r = check_layout(lay, d);
  if (r) return r;
  if ((r = check_cache(d, c))) return r;
  if ((r = check_range(d, layer0, n_layers))) return r;
  if (T < 0 || (T > 0 && (!k || !v || !pos))) return SSA_ERR_INVALID_ARG;
  if (!c->slab_scale || !c->slab_sum || !c->slab_cnt) return SSA_ERR_INVALID_ARG;
  if (T > 2147483647 / 2) return SSA_ERR_INVALID_ARG;
  cudaError_t e = launch_store(d, *c, layer0, n_layers, k, v, pos, T, status,
                               (cudaStream_t)stream);
  return e == cudaSuccess ? SSA_OK : fail_cuda(e);
}

int ssa_index_topk(const ssa_layout* lay, const ssa_cache* c, int layer0, int n_layers,
                   const void* q, const int32_t* block_table, const int32_t* seq_lens,
                   int32_t* sel, int32_t* n_sel, int32_t* scores_opt, int32_t* status,
                   void* ws, ssa_stream_t stream) {
  Dims d;
  int r = check_layout(lay, d);
  if (r) return r;
  if (!c || !c->slab) return SSA_ERR_INVALID_ARG;
  if ((r = check_range(d, layer0, n_layers))) return r;
  if (!q || !block_table || !seq_lens || !sel || !n_sel) return SSA_ERR_INVALID_ARG;
  if (!ws) return SSA_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(d);
  int32_t* scores = scores_opt ? scores_opt : at<int32_t>(ws, w.scores);
  cudaError_t e = launch_index_topk(d, *c, layer0, n_layers, q, block_table, seq_lens, scores,
                                    sel, n_sel, at<int32_t>(ws, w.idx_tickets), status,
                                    (cudaStream_t)stream);
  return e == cudaSuccess ? SSA_OK : fail_cuda(e);
}

static int ensure_impl(const ssa_layout* lay, const ssa_cache* c, int layer0, int n_layers,
                       const int32_t* sel, const int32_t* block_table, int32_t* miss_page_opt,
                       int32_t* miss_slot_opt, int32_t* n_miss_opt, int32_t* phys_opt,
                       int32_t* status, void* ws, ssa_stream_t stream) {
  Dims d;
  int r = check_layout(lay, d);
  if (r) return r;
  if ((r = check_cache(d, c))) return r;
  if ((r = check_range(d, layer0, n_layers))) return r;
  if (!sel || !block_table) return SSA_ERR_INVALID_ARG;
  const long long need = (long long)d.B * d.W < d.Lp ? (long long)d.B * d.W : d.Lp;
  if (d.S < need) return SSA_ERR_POOL_TOO_SMALL;
  if (!ws && (!miss_page_opt || !miss_slot_opt || !n_miss_opt)) return SSA_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(d);
  int32_t* mp = miss_page_opt ? miss_page_opt : at<int32_t>(ws, w.miss_page);
  int32_t* ms = miss_slot_opt ? miss_slot_opt : at<int32_t>(ws, w.miss_slot);
  int32_t* nm = n_miss_opt ? n_miss_opt : at<int32_t>(ws, w.n_miss);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_ensure_state(d, *c, layer0, n_layers, sel, block_table, mp, ms, nm,
                                      phys_opt, status, s);
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch_miss_copy(d, *c, layer0, n_layers, mp, ms, nm, status, s);
  return e == cudaSuccess ? SSA_OK : fail_cuda(e);
}

int ssa_ensure_resident(const ssa_layout* lay, const ssa_cache* c, int layer0, int n_layers,
                        const int32_t* sel, const int32_t* block_table,
                        int32_t* miss_page_opt, int32_t* miss_slot_opt, int32_t* n_miss_opt,
                        int32_t* status, void* ws, ssa_stream_t stream) {
  return ensure_impl(lay, c, layer0, n_layers, sel, block_table, miss_page_opt, miss_slot_opt,
                     n_miss_opt, nullptr, status, ws, stream);
}

int ssa_ensure_remap(const ssa_layout* lay, const ssa_cache* c, int layer0, int n_layers,
                     const int32_t* sel, const int32_t* block_table, int32_t* phys,
                     int32_t* miss_page_opt, int32_t* miss_slot_opt, int32_t* n_miss_opt,
                     int32_t* status, void* ws, ssa_stream_t stream) {
  if (!phys) return SSA_ERR_INVALID_ARG;
  return ensure_impl(lay, c, layer0, n_layers, sel, block_table, miss_page_opt, miss_slot_opt,
                     n_miss_opt, phys, status, ws, stream);
}

int ssa_ensure_remap_bind(const ssa_layout* lay, const ssa_cache* c, int layer0, int n_layers,
                          const int32_t* sel, const int32_t* block_table, int32_t* phys,
                          int32_t* miss_page, int32_t* miss_slot, int32_t* n_miss,
                          int32_t* status, ssa_stream_t stream) {
  Dims d;
  int r = check_layout(lay, d);
  if (r) return r;
  if ((r = check_cache(d, c))) return r;
  if ((r = check_range(d, layer0, n_layers))) return r;
  if (!sel || !block_table || !phys || !miss_page || !miss_slot || !n_miss)
    return SSA_ERR_INVALID_ARG;
  const long long need = (long long)d.B * d.W < d.Lp ? (long long)d.B * d.W : d.Lp;
  if (d.S < need) return SSA_ERR_POOL_TOO_SMALL;
  cudaError_t e = launch_ensure_state(d, *c, layer0, n_layers, sel, block_table, miss_page,
                                      miss_slot, n_miss, phys, status, (cudaStream_t)stream);
  return e == cudaSuccess ? SSA_OK : fail_cuda(e);
}

int ssa_fetch_misses(const ssa_layout* lay, const ssa_cache* c, int layer0, int n_layers,
                     const int32_t* miss_page, const int32_t* miss_slot, const int32_t* n_miss,
                     int32_t* status, ssa_stream_t stream) {
  Dims d;
  int r = check_layout(lay, d);
  if (r) return r;
  if ((r = check_cache(d, c))) return r;
  if ((r = check_range(d, layer0, n_layers))) return r;
  if (!miss_page || !miss_slot || !n_miss) return SSA_ERR_INVALID_ARG;
  if (!has_mirror(d, c)) return SSA_ERR_NO_MIRROR;
  cudaError_t e = launch_miss_copy(d, *c, layer0, n_layers, miss_page, miss_slot, n_miss, status,
                                   (cudaStream_t)stream);
  return e == cudaSuccess ? SSA_OK : fail_cuda(e);
}

int ssa_ensure_remap_deferred(const ssa_layout* lay, const ssa_cache* c, int layer0,
                              int n_layers, const int32_t* sel, const int32_t* block_table,
                              int32_t* phys, int32_t* miss_page_opt, int32_t* miss_slot_opt,
                              int32_t* n_miss_opt, int32_t* status, void* ws,
                              ssa_stream_t stream) {
  Dims d;
  int r = check_layout(lay, d);
  if (r) return r;
  if ((r = check_cache(d, c))) return r;
  if ((r = check_range(d, layer0, n_layers))) return r;
  if (!sel || !block_table || !phys) return SSA_ERR_INVALID_ARG;
  if (!has_mirror(d, c)) return SSA_ERR_NO_MIRROR;        // the attention fetches from it
  const long long need = (long long)d.B * d.W < d.Lp ? (long long)d.B * d.W : d.Lp;
  if (d.S < need) return SSA_ERR_POOL_TOO_SMALL;
  if (!ws && (!miss_page_opt || !miss_slot_opt || !n_miss_opt)) return SSA_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(d);
  int32_t* mp = miss_page_opt ? miss_page_opt : at<int32_t>(ws, w.miss_page);
  int32_t* ms = miss_slot_opt ? miss_slot_opt : at<int32_t>(ws, w.miss_slot);
  int32_t* nm = n_miss_opt ? n_miss_opt : at<int32_t>(ws, w.n_miss);
  cudaError_t e = launch_ensure_state_deferred(d, *c, layer0, n_layers, sel, block_table, mp, ms,
                                               nm, phys, status, (cudaStream_t)stream);
  return e == cudaSuccess ? SSA_OK : fail_cuda(e);
}

int ssa_ensure_remap_shared(const ssa_layout* lay, const ssa_cache* c, int layer0,
                            int n_layers, const int32_t* sel, const int32_t* block_table,
                            int32_t* phys, int32_t* miss_page_opt, int32_t* miss_slot_opt,
                            int32_t* n_miss_opt, int32_t* status, void* ws,
                            ssa_stream_t stream) {
  Dims d;
  int r = check_layout(lay, d);
  if (r) return r;
  if ((r = check_cache(d, c))) return r;
  if ((r = check_range(d, layer0, n_layers))) return r;
  if (!sel || !block_table || !phys) return SSA_ERR_INVALID_ARG;
  if (!ws && (!miss_page_opt || !miss_slot_opt || !n_miss_opt)) return SSA_ERR_INVALID_ARG;
  const long long entries = (long long)n_layers * d.B * d.W;
  if (entries > 16384) return SSA_ERR_UNSUPPORTED;      // the union is sorted in shared memory
  const long long need = entries < d.Lp ? entries : d.Lp;
  if (d.S < need) return SSA_ERR_POOL_TOO_SMALL;
  const WsLayout w = ws_layout(d);
  int32_t* mp = miss_page_opt ? miss_page_opt : at<int32_t>(ws, w.miss_page);
  int32_t* ms = miss_slot_opt ? miss_slot_opt : at<int32_t>(ws, w.miss_slot);
  int32_t* nm = n_miss_opt ? n_miss_opt : at<int32_t>(ws, w.n_miss);
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_ensure_state_shared(d, *c, layer0, n_layers, sel, block_table, mp, ms,
                                             nm, phys, status, s);
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch_miss_copy(d, *c, layer0, n_layers, mp, ms, nm, status, s, true);
  return e == cudaSuccess ? SSA_OK : fail_cuda(e);
}

int ssa_prefetch_pages(const ssa_layout* lay, const ssa_cache* c, int layer0, int n_layers,
                       const int32_t* scores, const int32_t* block_table, const int32_t* seq_lens,
                       int width, int32_t* fetch_page_opt, int32_t* fetch_slot_opt,
                       int32_t* n_fetch_opt, int32_t* status, void* ws, ssa_stream_t stream) {
  Dims d;
  int r = check_layout(lay, d);
  if (r) return r;
  if ((r = check_cache(d, c))) return r;
  if ((r = check_range(d, layer0, n_layers))) return r;
  if (!scores || !block_table || !seq_lens || !ws) return SSA_ERR_INVALID_ARG;
  if (width < 1 || width > d.W) return SSA_ERR_INVALID_ARG;
  const long long need = (long long)d.B * d.W < d.Lp ? (long long)d.B * d.W : d.Lp;
  if (d.S < need) return SSA_ERR_POOL_TOO_SMALL;
  const WsLayout w = ws_layout(d);
  int32_t* cand = at<int32_t>(ws, w.pf_cand);
  int32_t* mp = fetch_page_opt ? fetch_page_opt : at<int32_t>(ws, w.pf_miss_page);
  int32_t* ms = fetch_slot_opt ? fetch_slot_opt : at<int32_t>(ws, w.pf_miss_slot);
  int32_t* nm = n_fetch_opt ? n_fetch_opt : at<int32_t>(ws, w.pf_n_miss);
  cudaStream_t s = (cudaStream_t)stream;
  // the candidates: the selection rule with k = width - 1 over the step's scores
  Dims dw = d;
  dw.k = width - 1;
  dw.W = width;
  cudaError_t e = launch_topk_select(dw, n_layers, scores, seq_lens, cand,
                                     at<int32_t>(ws, w.pf_ncand), status, s);
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch_preload_state(d, *c, layer0, n_layers, cand, width, block_table, mp, ms, nm, status,
                           s);
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch_miss_copy(d, *c, layer0, n_layers, mp, ms, nm, status, s);
  return e == cudaSuccess ? SSA_OK : fail_cuda(e);
}

int ssa_remap_block_table(const ssa_layout* lay, const ssa_cache* c, int layer0, int n_layers,
                          const int32_t* sel, const int32_t* block_table, int32_t* phys,
                          int32_t* status, ssa_stream_t stream) {
  Dims d;
  int r = check_layout(lay, d);
  if (r) return r;
  if (!c || !c->slot_of) return SSA_ERR_INVALID_ARG;
  if ((r = check_range(d, layer0, n_layers))) return r;
  if (!sel || !block_table || !phys) return SSA_ERR_INVALID_ARG;
  cudaError_t e = launch_remap(d, *c, layer0, n_layers, sel, block_table, phys, status,
                               (cudaStream_t)stream);
  return e == cudaSuccess ? SSA_OK : fail_cuda(e);
}

// mode: 0 resident (phys), 1 host tail (block_table, slot_of), 2 fetch (phys
// with deferred misses marked, block_table)
static int decode_impl(const ssa_layout* lay, const ssa_cache* c, int layer0, int n_layers,
                       const void* q, const int32_t* sel, const int32_t* phys,
                       const int32_t* block_table, const int32_t* seq_lens, float sm_scale,
                       void* out, int32_t* status, void* ws, ssa_stream_t stream, int mode) {
  Dims d;
  int r = check_layout(lay, d);
  if (r) return r;
  if (!c || !c->k_pool || !c->v_pool || (d.fp8 && (!c->k_scale || !c->v_scale)))
    return SSA_ERR_INVALID_ARG;
  if ((r = check_range(d, layer0, n_layers))) return r;
  const bool host_tail = mode == 1, fetch = mode == 2;
  if (!q || !sel || (!phys && !host_tail) || !seq_lens || !out) return SSA_ERR_INVALID_ARG;
  if ((host_tail || fetch) && !block_table) return SSA_ERR_INVALID_ARG;
  if (!ws) return SSA_ERR_INVALID_ARG;
  if (host_tail || fetch) {
    if (host_tail && !c->slot_of) return SSA_ERR_INVALID_ARG;
    if (!mirror_consistent(d, c) || !has_mirror(d, c)) return SSA_ERR_NO_MIRROR;
  }
  const WsLayout w = ws_layout(d);
  DecodeArgs a{};
  a.d = &d;
  a.c = c;
  a.layer0 = layer0;
  a.n_layers = n_layers;
  a.num_sms = num_sms();
  a.q = q;
  a.sel = sel;
  a.phys = phys;
  a.seq_lens = seq_lens;
  a.sm_scale = sm_scale;
  a.out = out;
  a.part_o = at<float>(ws, w.part_o);
  a.part_ml = at<float>(ws, w.part_ml);
  a.tickets = at<int32_t>(ws, w.tickets);
  a.status = status;
  a.host_tail = host_tail ? 1 : 0;
  a.fetch = fetch ? 1 : 0;
  a.bt = block_table;
  cudaError_t e = launch_decode(a, (cudaStream_t)stream);
  return e == cudaSuccess ? SSA_OK : fail_cuda(e);
}

int ssa_sparse_paged_decode(const ssa_layout* lay, const ssa_cache* c, int layer0, int n_layers,
                            const void* q, const int32_t* sel, const int32_t* phys,
                            const int32_t* seq_lens, float sm_scale, void* out,
                            int32_t* status, void* ws, ssa_stream_t stream) {
  return decode_impl(lay, c, layer0, n_layers, q, sel, phys, nullptr, seq_lens, sm_scale, out,
                     status, ws, stream, 0);
}

int ssa_sparse_paged_decode_fetch(const ssa_layout* lay, const ssa_cache* c, int layer0,
                                  int n_layers, const void* q, const int32_t* sel,
                                  const int32_t* phys, const int32_t* block_table,
                                  const int32_t* seq_lens, float sm_scale, void* out,
                                  int32_t* status, void* ws, ssa_stream_t stream) {
  return decode_impl(lay, c, layer0, n_layers, q, sel, phys, block_table, seq_lens, sm_scale,
                     out, status, ws, stream, 2);
}

int ssa_sparse_paged_decode_host_tail(const ssa_layout* lay, const ssa_cache* c, int layer0,
                                      int n_layers, const void* q, const int32_t* sel,
                                      const int32_t* block_table, const int32_t* seq_lens,
                                      float sm_scale, void* out, int32_t* status, void* ws,
                                      ssa_stream_t stream) {
  if (!block_table) return SSA_ERR_INVALID_ARG;
  return decode_impl(lay, c, layer0, n_layers, q, sel, nullptr, block_table, seq_lens, sm_scale,
                     out, status, ws, stream, 1);
}

const char* ssa_status_str(int code) {
  switch (code) {
    case SSA_OK: return "ok";
    case SSA_ERR_INVALID_ARG: return "invalid argument (null pointer, layer range or layout field)";
    case SSA_ERR_POOL_TOO_SMALL: return "pool_slots < min(batch * max_sel, logical_pages)";
    case SSA_ERR_UNSUPPORTED: return "unsupported layout (dtype, page size, head_dim, GQA group)";
    case SSA_ERR_NO_MIRROR: return "host mirror pointers incomplete";
    case SSA_ERR_CUDA: return "CUDA launch failed (see ssa_last_cuda_error)";
    case SSA_ERR_SCRATCH_LIMIT:
      return "n_layers * batch * max_pages exceeds the static score scratch (SSA_STATIC_SCORE_ENTRIES)";
    default: break;
  }
  if (code > 0) {
    static thread_local char buf[256];
    buf[0] = 0;
    const char* names[] = {"drop", "bad_id", "miss_no_mirror", "unresolved", "bad_pos",
                           "timeout", "internal"};
    for (int i = 0; i < 7; ++i)
      if (code & (1 << i)) {
        if (buf[0]) strncat(buf, "|", sizeof(buf) - strlen(buf) - 1);
        strncat(buf, names[i], sizeof(buf) - strlen(buf) - 1);
      }
    return buf;
  }
  return "unknown status";
}

int ssa_last_cuda_error(void) { return g_last_cuda_error; }

long long ssa_launch_count(void) { return g_launches; }

}  // extern "C"
