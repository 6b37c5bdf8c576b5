// Internal interfaces between the host entry points (exq_api.cu) and the
// kernel translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "exq.h"

namespace exq {

// device error codes recorded by kernels (OR-ed into a per-module word)
enum : unsigned {
  kDevErrTimeout = 1u,      // a bounded wait gave up
  kDevErrBadSegment = 2u,   // an EXL2 segment width outside {2,3,4,5,6,8} or past the end
  kDevErrBadPerm = 4u,      // a permutation entry outside [0, K)
};

// failure-detection test hook (exq_testing.h): 0 = off, else the wait bound
// (polling rounds) for launches whose producer is to issue nothing
int testing_starve_rounds();

struct DeviceInfo {
  int sm_count = 0;
  int max_smem_optin = 0;
  int cc_major = 0, cc_minor = 0;
};

// queried once per device, cached (host-only, thread-safe)
const DeviceInfo& device_info(int device);

// cuTensorMapEncodeTiled from the driver, looked up once (nullptr if absent)
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled tensor_map_encoder();

// A 2-D tiled tensor map without swizzle: dims {inner, outer} elements, the
// outer stride in bytes, box {box_inner, box_outer}; elements outside the
// tensor read as zero; `promotion` sets how much L2 fetches around each
// access. False if the driver rejects it.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner, uint64_t outer,
               uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapL2promotion promotion = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);

// n layers (1..EXQ_GEMV_MAX_LAYERS) of one format and K that share x
exq_status launch_gemv(const exq_weight* w, int n, const uint16_t* x, int M, uint16_t* const* y, void* workspace,
                       size_t ws_bytes, cudaStream_t stream);
size_t gemv_workspace_bytes(const exq_weight* w, int n, int M);
exq_status launch_dequant(const exq_weight& w, uint16_t* W_out, cudaStream_t stream);
// n layers (1..EXQ_GEMM_MAX_LAYERS) of one format and K that share x
exq_status launch_gemm(const exq_weight* w, int n, const uint16_t* x, int M, uint16_t* const* y, void* workspace,
                       size_t ws_bytes, cudaStream_t stream);
size_t gemm_workspace_bytes(const exq_weight* w, int n, int M);
// the act-order part of it: M * K * 2 rounded up to 256 bytes, 0 without a permutation
size_t gemm_gather_bytes(const exq_weight& w, int M);
// exq_gemm with the library's static scratch array as the workspace
exq_status launch_gemm_noalloc(const exq_weight& w, const uint16_t* x, int M, uint16_t* y, cudaStream_t stream);

// quantized KV cache codec (D in {64, 128, 256}, b in {4, 6, 8}, checked by the caller)
exq_status launch_kv_quantize(const uint16_t* x, long long n_groups, int D, int b, uint32_t* codes,
                              uint16_t* scales, cudaStream_t stream);
exq_status launch_kv_dequantize(const uint32_t* codes, const uint16_t* scales, long long n_groups, int D, int b,
                                uint16_t* x_out, cudaStream_t stream);

// EXL2 conversion: RTN quantiser into the EXL2 layout, and the error table
exq_status launch_rtn_quantize(const uint16_t* W, const int32_t* perm, int K, int N, const uint32_t* seg_off,
                               int n_word_rows, uint32_t* qweight, uint16_t* scales, cudaStream_t stream);
exq_status launch_rtn_measure(const uint16_t* W, const int32_t* perm, int K, int N, float* err, void* workspace,
                              cudaStream_t stream);
size_t measure_workspace_bytes(int K, int N);

// read-and-clear of each module's device error word (stream-ordered copy +
// synchronise); returns the OR of the codes or ~0u on a CUDA failure
unsigned take_gemv_errors(cudaStream_t stream);
unsigned take_dequant_errors(cudaStream_t stream);
unsigned take_gemm_errors(cudaStream_t stream);
unsigned take_convert_errors(cudaStream_t stream);

}  // namespace exq
