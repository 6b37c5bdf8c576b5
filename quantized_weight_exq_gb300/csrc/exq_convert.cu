// EXL2 conversion on the GPU without calibration data: round-to-nearest
// quantisation of an fp16 weight into the EXL2 layout, and the table of
// weight-space errors per (segment, width) that a bits solve consumes.
//
// The ExLlamaV2 blog post ("ExLlamaV2: The fastest inference engine for
// quantized Llama/HF models", "How the EXL2 Quantization Pipeline Works Under
// the Hood") measures each layer at every width on calibration text (Step 1),
// solves for a width per group at a target bpw (Step 2) and quantises
// (Step 3). Without calibration data the measurement here is the squared
// error of the weights themselves. The quantiser is symmetric RTN per
// (32-row segment, column), qmax = 2^(b-1) - 1:
//   s = fp16_RN(fp32_RN(amax / qmax)),
//   q = clamp(rint(fp32_RN(w / s)), -qmax - 1, qmax)  (0 where s = 0),
//   stored code u = q + 2^(b-1)  (the EXL2 zero), w_hat = fp16_RN(q s).
//
// One thread per (segment, column). A block first copies its 32 x 256 tile of
// W (rows perm[32 s + i]) into shared memory with 16-byte loads, 512
// contiguous bytes per row; each thread then takes its column's 32 values from
// there. Codes leave as the segment's b word rows.
#include "exq_device.cuh"
#include "exq_internal.h"

namespace exq {
namespace {

__device__ unsigned g_convert_err;

constexpr int kThreads = 256;  // columns per block

// The block's tile: 32 rows x 256 columns of fp16 into shared memory (each
// thread moves four 16-byte vectors; columns past N are left unset), then the
// calling thread's column as fp32. Every thread of the block must call it.
__device__ __forceinline__ void load_segment(const uint16_t* __restrict__ W, const int32_t* __restrict__ perm, int K,
                                             int N, int seg, int n0, uint16_t (*tile)[kThreads], float (&v)[32]) {
  const int c = threadIdx.x & 31;  // 16-byte vector of the row: columns n0 + 8c .. + 7
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = (threadIdx.x >> 5) + 8 * k;
    const int j = seg * 32 + r;
    const int row = perm ? __ldg(perm + j) : j;
    const bool ok = static_cast<unsigned>(row) < static_cast<unsigned>(K);
    if (!ok && c == 0) atomicOr(&g_convert_err, kDevErrBadPerm);
    uint4 q = make_uint4(0u, 0u, 0u, 0u);
    if (ok && n0 + 8 * c < N) q = __ldg(reinterpret_cast<const uint4*>(W + static_cast<size_t>(row) * N + n0 + 8 * c));
    *reinterpret_cast<uint4*>(&tile[r][8 * c]) = q;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __half2float(__ushort_as_half(tile[i][threadIdx.x]));
}

// scale (fp16 bits) and codes q (signed) of one width
template <int B>
__device__ __forceinline__ uint16_t rtn(const float (&v)[32], int (&q)[32]) {
  constexpr int kQmax = (1 << (B - 1)) - 1;
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const __half s16 = __float2half_rn(__fdiv_rn(amax, static_cast<float>(kQmax)));
  const float s = __half2float(s16);
  const float inv = s != 0.f ? __frcp_rn(s) : 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) q[i] = s != 0.f ? max(-kQmax - 1, min(kQmax, round_quotient(v[i], s, inv))) : 0;
  return __half_as_ushort(s16);
}

template <int B>
__device__ __forceinline__ void quantize_store(const float (&v)[32], uint32_t* __restrict__ qw, size_t N, int n,
                                               uint16_t* __restrict__ scale) {
  int q[32];
  *scale = rtn<B>(v, q);
  // the column's stream: code i at bits [i B, i B + B), whole words out in order
  unsigned long long window = 0;
  int have = 0, word = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    window |= static_cast<unsigned long long>(q[i] + (1 << (B - 1))) << have;
    have += B;
    if (have >= 32) {
      qw[static_cast<size_t>(word++) * N + n] = static_cast<uint32_t>(window);
      window >>= 32;
      have -= 32;
    }
  }
}

__global__ void __launch_bounds__(kThreads)
    rtn_quantize_kernel(const uint16_t* __restrict__ W, const int32_t* __restrict__ perm, int K, int N,
                        const uint32_t* __restrict__ seg_off, int n_word_rows, uint32_t* __restrict__ qweight,
                        uint16_t* __restrict__ scales) {
  __shared__ __align__(16) uint16_t tile[32][kThreads];
  const int seg = blockIdx.y;
  const int n0 = blockIdx.x * kThreads, n = n0 + threadIdx.x;
  const uint32_t o0 = __ldg(seg_off + seg), o1 = __ldg(seg_off + seg + 1);
  const int b = static_cast<int>(o1) - static_cast<int>(o0);
  const bool good = (b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8) &&
                    o1 <= static_cast<uint32_t>(n_word_rows);
  if (!good) {  // reported (block-uniform); the segment's rows are left untouched
    if (threadIdx.x == 0) atomicOr(&g_convert_err, kDevErrBadSegment);
    return;
  }
  float v[32];
  load_segment(W, perm, K, N, seg, n0, tile, v);
  if (n >= N) return;
  uint32_t* qw = qweight + static_cast<size_t>(o0) * N;
  uint16_t* sc = scales + static_cast<size_t>(seg) * N + n;
  switch (b) {
    case 2: quantize_store<2>(v, qw, N, n, sc); break;
    case 3: quantize_store<3>(v, qw, N, n, sc); break;
    case 4: quantize_store<4>(v, qw, N, n, sc); break;
    case 5: quantize_store<5>(v, qw, N, n, sc); break;
    case 6: quantize_store<6>(v, qw, N, n, sc); break;
    default: quantize_store<8>(v, qw, N, n, sc); break;
  }
}

// sum over the segment's 32 values of (v - w_hat)^2 at width B
template <int B>
__device__ __forceinline__ float segment_error(const float (&v)[32]) {
  int q[32];
  const float s = __half2float(__ushort_as_half(rtn<B>(v, q)));
  float e = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float w_hat = __half2float(__float2half_rn(static_cast<float>(q[i]) * s));  // q s is exact in fp32
    const float d = v[i] - w_hat;
    e = fmaf(d, d, e);
  }
  return e;
}

// per (segment, block of 256 columns): the six error sums of the block's
// columns, added in a fixed order (warp shuffles, then warps in order)
__global__ void __launch_bounds__(kThreads)
    rtn_measure_kernel(const uint16_t* __restrict__ W, const int32_t* __restrict__ perm, int K, int N,
                       float* __restrict__ partial) {
  __shared__ float red[kThreads / 32][6];
  __shared__ __align__(16) uint16_t tile[32][kThreads];
  const int seg = blockIdx.y;
  const int n0 = blockIdx.x * kThreads, n = n0 + threadIdx.x;
  float e[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float v[32];
  load_segment(W, perm, K, N, seg, n0, tile, v);
  if (n < N) {
    e[0] = segment_error<2>(v);
    e[1] = segment_error<3>(v);
    e[2] = segment_error<4>(v);
    e[3] = segment_error<5>(v);
    e[4] = segment_error<6>(v);
    e[5] = segment_error<8>(v);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < 6; ++k) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) e[k] += __shfl_down_sync(0xffffffffu, e[k], d);
    if (lane == 0) red[warp][k] = e[k];
  }
  __syncthreads();
  if (threadIdx.x < 6) {
    float t = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) t += red[w][threadIdx.x];
    partial[(static_cast<size_t>(seg) * gridDim.x + blockIdx.x) * 6 + threadIdx.x] = t;
  }
}

// err[seg][k] = the column blocks' partial sums added in block order
__global__ void measure_finish_kernel(const float* __restrict__ partial, int S, int blocks, float* __restrict__ err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;  // seg * 6 + k
  if (i >= S * 6) return;
  const int seg = i / 6, k = i - seg * 6;
  float t = 0.f;
  for (int c = 0; c < blocks; ++c) t += partial[(static_cast<size_t>(seg) * blocks + c) * 6 + k];
  err[i] = t;
}

}  // namespace

size_t measure_workspace_bytes(int K, int N) {
  const size_t blocks = (static_cast<size_t>(N) + kThreads - 1) / kThreads;
  return static_cast<size_t>(K / 32) * blocks * 6 * sizeof(float);
}

exq_status launch_rtn_quantize(const uint16_t* W, const int32_t* perm, int K, int N, const uint32_t* seg_off,
                               int n_word_rows, uint32_t* qweight, uint16_t* scales, cudaStream_t stream) {
  const dim3 grid((N + kThreads - 1) / kThreads, K / 32);
  rtn_quantize_kernel<<<grid, kThreads, 0, stream>>>(W, perm, K, N, seg_off, n_word_rows, qweight, scales);
  return cudaGetLastError() == cudaSuccess ? EXQ_OK : EXQ_ERR_CUDA;
}

exq_status launch_rtn_measure(const uint16_t* W, const int32_t* perm, int K, int N, float* err, void* workspace,
                              cudaStream_t stream) {
  const int blocks = (N + kThreads - 1) / kThreads, S = K / 32;
  float* partial = static_cast<float*>(workspace);
  rtn_measure_kernel<<<dim3(blocks, S), kThreads, 0, stream>>>(W, perm, K, N, partial);
  if (cudaGetLastError() != cudaSuccess) return EXQ_ERR_CUDA;
  measure_finish_kernel<<<(S * 6 + 255) / 256, 256, 0, stream>>>(partial, S, blocks, err);
  return cudaGetLastError() == cudaSuccess ? EXQ_OK : EXQ_ERR_CUDA;
}

unsigned take_convert_errors(cudaStream_t stream) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_convert_err, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return ~0u;
  if (cudaMemcpyToSymbolAsync(g_convert_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
      cudaSuccess)
    return ~0u;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
  return v;
}

}  // namespace exq
