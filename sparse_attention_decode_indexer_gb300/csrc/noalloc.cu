// noalloc.cu -- ssa_index_topk_static_scratch: the indexer + top-k selection
// with its score scratch in a fixed device array that is part of the library.
//
// For callers that cannot allocate device memory at all -- a plugin running
// inside a host program that owns every device allocation, or a serving
// loop that must not allocate once it is up -- and so cannot provide the
// workspace that ssa_index_topk takes.  Everything else (inputs, outputs,
// the cache) is still the caller's.
//
// The scratch is one file-scope __device__ array of SSA_STATIC_SCORE_ENTRIES
// int32 scores (4 MiB), held by every GPU that loads the library until the
// process exits.  Host code may not use the array's name as a device
// address (on the host it names a stand-in), so the address is fetched once
// per device with cudaGetSymbolAddress and cached.  All calls share the
// array: calls whose kernels overlap on the GPU race on it.  Nothing in it
// needs clearing between calls: the score kernel writes every entry the
// select kernel reads.
#include <mutex>

#include "internal.h"

namespace {

__device__ __align__(256) int32_t g_score_scratch[SSA_STATIC_SCORE_ENTRIES];

constexpr int kMaxDevices = 64;
int32_t* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_score_scratch on the current device (set up on first use).
cudaError_t scratch_for_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_score_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int ssa_index_topk_static_scratch(const ssa_layout* lay, const ssa_cache* c,
                                             int layer0, int n_layers, const void* q,
                                             const int32_t* block_table,
                                             const int32_t* seq_lens, int32_t* sel,
                                             int32_t* n_sel, int32_t* status,
                                             ssa_stream_t stream) {
  ssa::Dims d;
  int r = ssa::validate_layout(lay, d);
  if (r) return r;
  if (!c || !c->slab) return SSA_ERR_INVALID_ARG;
  if (layer0 < 0 || n_layers < 1 || layer0 + n_layers > d.Lyr) return SSA_ERR_INVALID_ARG;
  if (!q || !block_table || !seq_lens || !sel || !n_sel) return SSA_ERR_INVALID_ARG;
  if ((unsigned long long)n_layers * d.B * d.nmax > SSA_STATIC_SCORE_ENTRIES)
    return SSA_ERR_SCRATCH_LIMIT;
  int32_t* scores = nullptr;
  cudaError_t e = scratch_for_current_device(&scores);
  if (e != cudaSuccess) return ssa::record_cuda_error(e);
  cudaStream_t s = (cudaStream_t)stream;
  e = ssa::launch_index_scores(d, *c, layer0, n_layers, q, block_table, seq_lens, scores,
                               status, s);
  if (e != cudaSuccess) return ssa::record_cuda_error(e);
  e = ssa::launch_topk_select(d, n_layers, scores, seq_lens, sel, n_sel, status, s);
  return e == cudaSuccess ? SSA_OK : ssa::record_cuda_error(e);
}
