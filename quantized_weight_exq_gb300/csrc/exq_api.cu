// Host entry points of libexq: argument checks, dispatch, status codes.
// Every check here runs before any launch and has no side effects.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "exq_internal.h"
#include "exq_testing.h"

namespace exq {

const DeviceInfo& device_info(int device) {
  constexpr int kMaxDevices = 64;
  static DeviceInfo infos[kMaxDevices];
  static std::once_flag once[kMaxDevices];
  static DeviceInfo none;
  if (device < 0 || device >= kMaxDevices) return none;
  std::call_once(once[device], [device] {
    DeviceInfo d;
    cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device);
    cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, device);
    infos[device] = d;
  });
  return infos[device];
}

EncodeTiled tensor_map_encoder() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner, uint64_t outer,
               uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapL2promotion promotion) {
  EncodeTiled enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t gdim[2] = {inner, outer};
  const cuuint64_t gstride[1] = {outer_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return enc(map, type, 2, const_cast<void*>(base), gdim, gstride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, promotion,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
std::atomic<int> g_starve_rounds{0};
}  // namespace

int testing_starve_rounds() { return g_starve_rounds.load(std::memory_order_relaxed); }

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// structural checks of a layer descriptor (host-visible fields only)
exq_status check_weight(const exq_weight* w) {
  if (!w) return EXQ_ERR_INVALID_ARG;
  if (w->K <= 0 || w->N <= 0 || w->N % 8 || w->K % 32) return EXQ_ERR_INVALID_ARG;
  if (!w->qweight || !aligned16(w->qweight)) return EXQ_ERR_INVALID_ARG;
  if (w->perm && !aligned16(w->perm)) return EXQ_ERR_INVALID_ARG;
  // fp16 scales, or (EXL2 two-level) codes and column maxima instead
  const bool two_level = w->format == EXQ_FMT_EXL2_QSCALE;
  if (two_level) {
    if (w->scales || !w->q_scale || !w->q_scale_max || !aligned16(w->q_scale) || !aligned16(w->q_scale_max))
      return EXQ_ERR_INVALID_ARG;
  } else {
    if (!w->scales || !aligned16(w->scales) || w->q_scale || w->q_scale_max) return EXQ_ERR_INVALID_ARG;
  }
  if (w->format == EXQ_FMT_GPTQ4) {
    if (w->group_size <= 0 || w->group_size % 32 || w->K % w->group_size) return EXQ_ERR_INVALID_ARG;
    if (w->n_groups != w->K / w->group_size || w->n_word_rows != w->K / 8) return EXQ_ERR_INVALID_ARG;
    if (!w->qzeros || !aligned16(w->qzeros) || w->seg_word_off) return EXQ_ERR_INVALID_ARG;
  } else if (w->format == EXQ_FMT_EXL2 || two_level) {
    if (w->group_size != 32 || w->n_groups != w->K / 32) return EXQ_ERR_INVALID_ARG;
    if (w->n_word_rows < 2 * w->n_groups || w->n_word_rows > 8 * w->n_groups) return EXQ_ERR_INVALID_ARG;
    if (!w->seg_word_off || w->qzeros) return EXQ_ERR_INVALID_ARG;
  } else {
    return EXQ_ERR_INVALID_ARG;
  }
  return EXQ_OK;
}

// layers of one exq_gemv_multi call: each valid, one format, one K, one group size
exq_status check_group(const exq_weight* w, int n) {
  if (!w || n < 1 || n > EXQ_GEMV_MAX_LAYERS) return EXQ_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    const exq_status st = check_weight(&w[i]);
    if (st != EXQ_OK) return st;
    if (w[i].format != w[0].format || w[i].K != w[0].K || w[i].group_size != w[0].group_size)
      return EXQ_ERR_INVALID_ARG;
  }
  return EXQ_OK;
}

int current_cc() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  const DeviceInfo& di = device_info(dev);
  return di.cc_major * 10 + di.cc_minor;
}

}  // namespace
}  // namespace exq

using namespace exq;

extern "C" exq_status exq_dequant(const exq_weight* w, uint16_t* W_out, void* stream) {
  const exq_status st = check_weight(w);
  if (st != EXQ_OK) return st;
  if (!W_out || !aligned16(W_out)) return EXQ_ERR_INVALID_ARG;
  if (current_cc() < 100) return EXQ_ERR_CUDA;
  return launch_dequant(*w, W_out, static_cast<cudaStream_t>(stream));
}

extern "C" size_t exq_gemv_workspace_size(const exq_weight* w, int32_t M) {
  if (check_weight(w) != EXQ_OK || M < 1 || M > 16) return 0;
  return gemv_workspace_bytes(w, 1, M);
}

extern "C" exq_status exq_gemv(const exq_weight* w, const uint16_t* x, int32_t M, uint16_t* y, void* workspace,
                               size_t ws_bytes, void* stream) {
  const exq_status st = check_weight(w);
  if (st != EXQ_OK) return st;
  if (!x || !y || !aligned16(x) || !aligned16(y) || M < 1) return EXQ_ERR_INVALID_ARG;
  if (M > 16) return EXQ_ERR_UNSUPPORTED;
  if (current_cc() < 100) return EXQ_ERR_CUDA;
  return launch_gemv(w, 1, x, M, &y, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" size_t exq_gemv_multi_workspace_size(const exq_weight* w, int32_t n, int32_t M) {
  if (check_group(w, n) != EXQ_OK || M < 1 || M > 16) return 0;
  return gemv_workspace_bytes(w, n, M);
}

extern "C" exq_status exq_gemv_multi(const exq_weight* w, int32_t n, const uint16_t* x, int32_t M,
                                     uint16_t* const* y, void* workspace, size_t ws_bytes, void* stream) {
  const exq_status st = check_group(w, n);
  if (st != EXQ_OK) return st;
  if (!x || !y || !aligned16(x) || M < 1) return EXQ_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!y[i] || !aligned16(y[i])) return EXQ_ERR_INVALID_ARG;
  if (M > 16) return EXQ_ERR_UNSUPPORTED;
  if (current_cc() < 100) return EXQ_ERR_CUDA;
  return launch_gemv(w, n, x, M, y, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" size_t exq_gemm_workspace_size(const exq_weight* w, int32_t M) {
  if (check_weight(w) != EXQ_OK || M < 1) return 0;
  return gemm_workspace_bytes(w, 1, M);
}

extern "C" size_t exq_gemm_multi_workspace_size(const exq_weight* w, int32_t n, int32_t M) {
  if (n > EXQ_GEMM_MAX_LAYERS || check_group(w, n) != EXQ_OK || M < 1) return 0;
  return gemm_workspace_bytes(w, n, M);
}

extern "C" exq_status exq_gemm_multi(const exq_weight* w, int32_t n, const uint16_t* x, int32_t M,
                                     uint16_t* const* y, void* workspace, size_t ws_bytes, void* stream) {
  if (n > EXQ_GEMM_MAX_LAYERS) return EXQ_ERR_INVALID_ARG;
  const exq_status st = check_group(w, n);
  if (st != EXQ_OK) return st;
  if (!x || !y || !aligned16(x) || M < 1) return EXQ_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    if (!y[i] || !aligned16(y[i])) return EXQ_ERR_INVALID_ARG;
    if (w[i].K % 64 || w[i].N % 128) return EXQ_ERR_UNSUPPORTED;
  }
  const size_t need = gemm_workspace_bytes(w, n, M);
  if (need && (!workspace || ws_bytes < need || !aligned16(workspace))) return EXQ_ERR_INVALID_ARG;
  if (current_cc() < 100) return EXQ_ERR_CUDA;
  return launch_gemm(w, n, x, M, y, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" exq_status exq_gemm(const exq_weight* w, const uint16_t* x, int32_t M, uint16_t* y, void* workspace,
                               size_t ws_bytes, void* stream) {
  const exq_status st = check_weight(w);
  if (st != EXQ_OK) return st;
  if (!x || !y || !aligned16(x) || !aligned16(y) || M < 1) return EXQ_ERR_INVALID_ARG;
  const size_t need = gemm_workspace_bytes(w, 1, M);
  if (need && (!workspace || ws_bytes < need || !aligned16(workspace))) return EXQ_ERR_INVALID_ARG;
  if (current_cc() < 100) return EXQ_ERR_CUDA;
  return launch_gemm(w, 1, x, M, &y, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

extern "C" exq_status exq_gemm_noalloc(const exq_weight* w, const uint16_t* x, int32_t M, uint16_t* y,
                                       void* stream) {
  const exq_status st = check_weight(w);
  if (st != EXQ_OK) return st;
  if (!x || !y || !aligned16(x) || !aligned16(y) || M < 1) return EXQ_ERR_INVALID_ARG;
  if (gemm_gather_bytes(*w, M) > EXQ_NOALLOC_SCRATCH_BYTES) return EXQ_ERR_UNSUPPORTED;
  if (current_cc() < 100) return EXQ_ERR_CUDA;
  return launch_gemm_noalloc(*w, x, M, y, static_cast<cudaStream_t>(stream));
}

namespace {
// EXQ_OK with `empty` set: nothing to do (n_groups == 0; the pointers are not used)
exq_status check_kv(const void* a, const void* b, const void* c, long long n_groups, int D, int bits, bool& empty) {
  if (n_groups < 0) return EXQ_ERR_INVALID_ARG;
  if ((D != 64 && D != 128 && D != 256) || (bits != 4 && bits != 6 && bits != 8)) return EXQ_ERR_UNSUPPORTED;
  empty = n_groups == 0;
  if (empty) return EXQ_OK;
  if (!a || !b || !c || !aligned16(a) || !aligned16(b) || !aligned16(c)) return EXQ_ERR_INVALID_ARG;
  return EXQ_OK;
}
}  // namespace

extern "C" exq_status exq_kv_quantize(const uint16_t* x, int64_t n_groups, int32_t D, int32_t bits, uint32_t* codes,
                                      uint16_t* scales, void* stream) {
  bool empty = false;
  const exq_status st = check_kv(x, codes, scales, n_groups, D, bits, empty);
  if (st != EXQ_OK || empty) return st;
  if (current_cc() < 100) return EXQ_ERR_CUDA;
  return launch_kv_quantize(x, n_groups, D, bits, codes, scales, static_cast<cudaStream_t>(stream));
}

extern "C" exq_status exq_kv_dequantize(const uint32_t* codes, const uint16_t* scales, int64_t n_groups, int32_t D,
                                        int32_t bits, uint16_t* x_out, void* stream) {
  bool empty = false;
  const exq_status st = check_kv(codes, scales, x_out, n_groups, D, bits, empty);
  if (st != EXQ_OK || empty) return st;
  if (current_cc() < 100) return EXQ_ERR_CUDA;
  return launch_kv_dequantize(codes, scales, n_groups, D, bits, x_out, static_cast<cudaStream_t>(stream));
}

namespace {
exq_status check_convert(const uint16_t* W, const int32_t* perm, int K, int N) {
  if (!W || !aligned16(W) || (perm && !aligned16(perm))) return EXQ_ERR_INVALID_ARG;
  if (K <= 0 || N <= 0 || K % 32 || N % 8) return EXQ_ERR_INVALID_ARG;
  return EXQ_OK;
}
}  // namespace

extern "C" exq_status exq_quantize_exl2(const uint16_t* W, const int32_t* perm, int32_t K, int32_t N,
                                        const uint32_t* seg_word_off, int32_t n_word_rows, uint32_t* qweight_out,
                                        uint16_t* scales_out, void* stream) {
  const exq_status st = check_convert(W, perm, K, N);
  if (st != EXQ_OK) return st;
  if (!seg_word_off || !qweight_out || !scales_out || !aligned16(seg_word_off) || !aligned16(qweight_out) ||
      !aligned16(scales_out))
    return EXQ_ERR_INVALID_ARG;
  if (n_word_rows < 2 * (K / 32) || n_word_rows > 8 * (K / 32)) return EXQ_ERR_INVALID_ARG;
  if (current_cc() < 100) return EXQ_ERR_CUDA;
  return launch_rtn_quantize(W, perm, K, N, seg_word_off, n_word_rows, qweight_out, scales_out,
                             static_cast<cudaStream_t>(stream));
}

extern "C" size_t exq_measure_exl2_workspace_size(int32_t K, int32_t N) {
  if (K <= 0 || N <= 0 || K % 32 || N % 8) return 0;
  return measure_workspace_bytes(K, N);
}

extern "C" exq_status exq_measure_exl2(const uint16_t* W, const int32_t* perm, int32_t K, int32_t N, float* err_out,
                                       void* workspace, size_t ws_bytes, void* stream) {
  const exq_status st = check_convert(W, perm, K, N);
  if (st != EXQ_OK) return st;
  if (!err_out || !aligned16(err_out) || !workspace || !aligned16(workspace) ||
      ws_bytes < measure_workspace_bytes(K, N))
    return EXQ_ERR_INVALID_ARG;
  if (current_cc() < 100) return EXQ_ERR_CUDA;
  return launch_rtn_measure(W, perm, K, N, err_out, workspace, static_cast<cudaStream_t>(stream));
}

extern "C" const char* exq_status_string(exq_status s) {
  switch (s) {
    case EXQ_OK: return "ok";
    case EXQ_ERR_INVALID_ARG: return "invalid argument";
    case EXQ_ERR_UNSUPPORTED: return "unsupported shape or format";
    case EXQ_ERR_CUDA: return "CUDA error";
    case EXQ_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

extern "C" exq_status exq_get_last_device_error(void* stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const unsigned a = take_gemv_errors(s), b = take_dequant_errors(s), c = take_gemm_errors(s),
                 d = take_convert_errors(s);
  if (a == ~0u || b == ~0u || c == ~0u || d == ~0u) return EXQ_ERR_CUDA;
  const unsigned v = a | b | c | d;
  if (v & kDevErrTimeout) return EXQ_ERR_TIMEOUT;
  if (v & (kDevErrBadSegment | kDevErrBadPerm)) return EXQ_ERR_INVALID_ARG;
  return EXQ_OK;
}

extern "C" void exq_testing_starve(int32_t wait_rounds) {
  g_starve_rounds.store(wait_rounds > 0 ? wait_rounds : 0, std::memory_order_relaxed);
}
