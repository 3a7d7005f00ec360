// probe.cu -- ssa_host_read_probe: the host link's rate for reads that SMs
// issue themselves (16-byte loads from pinned host memory over unified
// addressing), the way the miss fetch reads the mirror.
//
// The copy engine's host-to-device rate (cudaMemcpyAsync) is one ceiling of
// the miss fetch; SM-driven loads are another, set by how many requests the
// SMs keep in flight and by the address translations of scattered pages.
// The probe copies a list of chunks (byte offsets into the source) into a
// contiguous device buffer, one group of CTAs per chunk, several 16-byte
// loads in flight per thread, so that a caller can time both a sequential
// stream and a miss-like scatter of page-sized chunks.
#include "common.cuh"
#include "internal.h"

namespace ssa {
namespace {

constexpr int kProbeThreads = 256;

template <int U>
__global__ void __launch_bounds__(kProbeThreads) host_read_probe_kernel(
    const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
    const int64_t* __restrict__ offsets, int chunk16) {
  const int chunk = blockIdx.y;
  const int64_t off = offsets[chunk];
  const uint4* s = reinterpret_cast<const uint4*>(src + off);
  uint4* d = reinterpret_cast<uint4*>(dst + (size_t)chunk * chunk16 * 16);
  uint4 buf[U];
  const int base = blockIdx.x * kProbeThreads * U + threadIdx.x;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int i = base + u * kProbeThreads;
    if (i < chunk16) buf[u] = s[i];
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int i = base + u * kProbeThreads;
    if (i < chunk16) d[i] = buf[u];
  }
}

}  // namespace
}  // namespace ssa

extern "C" int ssa_host_read_probe(const void* src, void* dst, const int64_t* offsets,
                                   int n_chunks, int chunk_bytes, int loads_per_thread,
                                   ssa_stream_t stream) {
  if (!src || !dst || !offsets || n_chunks < 1 || n_chunks > 65535 || chunk_bytes < 16 ||
      chunk_bytes % 16 != 0 || (reinterpret_cast<uintptr_t>(src) & 15) ||
      (reinterpret_cast<uintptr_t>(dst) & 15))
    return SSA_ERR_INVALID_ARG;
  if (loads_per_thread != 4 && loads_per_thread != 8 && loads_per_thread != 16)
    return SSA_ERR_INVALID_ARG;
  const int chunk16 = chunk_bytes / 16;
  const int per_cta = ssa::kProbeThreads * loads_per_thread;
  const dim3 grid((chunk16 + per_cta - 1) / per_cta, n_chunks);
  cudaStream_t s = (cudaStream_t)stream;
  const auto* sp = static_cast<const uint8_t*>(src);
  auto* dp = static_cast<uint8_t*>(dst);
  switch (loads_per_thread) {
    case 4: ssa::host_read_probe_kernel<4><<<grid, ssa::kProbeThreads, 0, s>>>(sp, dp, offsets, chunk16); break;
    case 8: ssa::host_read_probe_kernel<8><<<grid, ssa::kProbeThreads, 0, s>>>(sp, dp, offsets, chunk16); break;
    default: ssa::host_read_probe_kernel<16><<<grid, ssa::kProbeThreads, 0, s>>>(sp, dp, offsets, chunk16); break;
  }
  ssa::count_launch();
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SSA_OK : ssa::record_cuda_error(e);
}
