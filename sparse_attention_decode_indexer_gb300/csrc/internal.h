// internal.h -- launchers that the C ABI (api.cu) calls; one translation unit
// per stage of the decode step.  Host-side only; no torch types anywhere.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/ssa.h"

namespace ssa {

// Validated, derived view of an ssa_layout.
struct Dims {
  int P, Hq, Hkv, D, G, fp8, Lyr, Lp, S, B, nmax, k, W;
  size_t esz() const { return fp8 ? 1 : 2; }
  // bytes of one KV head of one page (K or V), and of a whole page (all heads)
  size_t head_page_bytes() const { return (size_t)P * D * esz(); }
  size_t page_bytes() const { return (size_t)Hkv * head_page_bytes(); }
  int max_selected() const { return k + 1 < nmax ? k + 1 : nmax; }
};

// Most CTAs one attention launch uses (one wave); the workspace holds two
// partial states per CTA.
int decode_max_ctas(const Dims& d, int num_sms);

// -- store.cu ---------------------------------------------------------------
cudaError_t launch_lru_init(const Dims& d, const ssa_cache& c, int identity, cudaStream_t s);
cudaError_t launch_store(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                         const void* k, const void* v, const int64_t* pos, int T,
                         int32_t* status, cudaStream_t s);

// -- index.cu ---------------------------------------------------------------
cudaError_t launch_index_scores(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                                const void* q, const int32_t* bt, const int32_t* seq_lens,
                                int32_t* scores, int32_t* status, cudaStream_t s);
// a1 + a2 fused: scores, then the last CTA per (layer, request) selects.
cudaError_t launch_index_topk(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                              const void* q, const int32_t* bt, const int32_t* seq_lens,
                              int32_t* scores, int32_t* sel, int32_t* n_sel, int32_t* tickets,
                              int32_t* status, cudaStream_t s);
cudaError_t launch_topk_select(const Dims& d, int n_layers, const int32_t* scores,
                               const int32_t* seq_lens, int32_t* sel, int32_t* n_sel,
                               int32_t* status, cudaStream_t s);

// -- ensure.cu --------------------------------------------------------------
// phys: null, or [n_layers][B][W] to receive the remapped table (a5 fused)
cudaError_t launch_ensure_state(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                                const int32_t* sel, const int32_t* bt, int32_t* miss_page,
                                int32_t* miss_slot, int32_t* n_miss, int32_t* phys,
                                int32_t* status, cudaStream_t s);
// The preload's state update: candidates cand [n_layers][B][width] (page
// indices, -1 padded) after a step's ensure; epoch clock - 1, the clock stays.
cudaError_t launch_preload_state(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                                 const int32_t* cand, int width, const int32_t* bt,
                                 int32_t* miss_page, int32_t* miss_slot, int32_t* n_miss,
                                 int32_t* status, cudaStream_t s);
// shared: one miss list (residency shared by the call's layers) copied into
// every layer's pool
cudaError_t launch_miss_copy(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                             const int32_t* miss_page, const int32_t* miss_slot,
                             const int32_t* n_miss, int32_t* status, cudaStream_t s,
                             bool shared = false);
// The ensure's state update and remap with the misses' fetch left to the
// attention: phys marks a page bound by this call as -2 - slot.
cudaError_t launch_ensure_state_deferred(const Dims& d, const ssa_cache& c, int layer0,
                                         int n_layers, const int32_t* sel, const int32_t* bt,
                                         int32_t* miss_page, int32_t* miss_slot, int32_t* n_miss,
                                         int32_t* phys, int32_t* status, cudaStream_t s);
// Residency shared by the layers of a call: one CTA ensures the union of the
// layers' selections sel [n_layers][B][W] on layer0's state; phys for every
// layer; the miss list [n_layers * B * W], its count n_miss[0].
cudaError_t launch_ensure_state_shared(const Dims& d, const ssa_cache& c, int layer0,
                                       int n_layers, const int32_t* sel, const int32_t* bt,
                                       int32_t* miss_page, int32_t* miss_slot, int32_t* n_miss,
                                       int32_t* phys, int32_t* status, cudaStream_t s);
cudaError_t launch_remap(const Dims& d, const ssa_cache& c, int layer0, int n_layers,
                         const int32_t* sel, const int32_t* bt, int32_t* phys,
                         int32_t* status, cudaStream_t s);

// -- decode.cu --------------------------------------------------------------
struct DecodeArgs {
  const Dims* d;
  const ssa_cache* c;
  int layer0, n_layers, num_sms;
  const void* q;
  const int32_t* sel;
  const int32_t* phys;
  const int32_t* seq_lens;
  float sm_scale;
  void* out;
  float* part_o;   // [decode_max_ctas][2][G][D]
  float* part_ml;  // [decode_max_ctas][2][G][2]
  int32_t* tickets;  // [units] piece counters (zero before the first call; left zero)
  int32_t* status;
  // host-tail mode: phys unused; pages resolved through slot_of, those
  // without a slot read from the mirror
  int host_tail;
  // fetch mode: phys entries -2 - slot are pages bound but not yet copied:
  // read from the mirror, used, and written into their slots
  int fetch;
  const int32_t* bt;  // [B][nmax]
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);

// Properties of the current device, queried once per device ordinal and
// cached (SM count; the most dynamic shared memory one CTA may opt in to).
constexpr int kMaxDevices = 64;
struct DeviceInfo { int sms, smem_optin; };
DeviceInfo current_device_info();
// The current device's ordinal, clamped to [0, kMaxDevices).
int current_device_ordinal();

// Counts every kernel launch the library enqueues (per host thread).
void count_launch(int n = 1);

// Layout validation shared by every entry point (fills the derived view).
int validate_layout(const ssa_layout* lay, Dims& d);

// Keeps a failed cudaError_t for ssa_last_cuda_error(); returns SSA_ERR_CUDA.
int record_cuda_error(cudaError_t e);

}  // namespace ssa
