// Prefill-sized fused quantized matmul (tcgen05). Placeholder until the
// tensor-memory kernel is in place: reports the shape as unsupported.
#include "exq_internal.h"

namespace exq {
namespace {
__device__ unsigned g_gemm_err;
}  // namespace

size_t gemm_workspace_bytes(const exq_weight& w, int M) {
  return w.perm ? static_cast<size_t>(M) * w.K * 2 : 0;
}

exq_status launch_gemm(const exq_weight&, const uint16_t*, int, uint16_t*, void*, size_t, cudaStream_t) {
  return EXQ_ERR_UNSUPPORTED;
}

unsigned take_gemm_errors(cudaStream_t stream) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_gemm_err, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return ~0u;
  if (cudaMemcpyToSymbolAsync(g_gemm_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return ~0u;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
  return v;
}

}  // namespace exq
