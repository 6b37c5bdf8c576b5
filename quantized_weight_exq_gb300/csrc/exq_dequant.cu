// Standalone dequantisation: W[perm[j]][n] = fp16_RN((q(j, n) - z) * s) for
// every stored row j -- the dense fp16 weight the ExLlamaV2 blog post
// ("ExLlamaV2: The fastest inference engine for quantized Llama/HF models",
// "Finding 2") describes as the "dequantize first" alternative to the fused
// kernel. Bit-exact: the subtraction is exact in fp16 and the only rounding
// is the final fp16 multiply.
//
// Work unit: one warp = one 32-row step x 64 columns. Lane (g = lane/4,
// t = lane%4) reads 8 adjacent columns (two 128-bit vectors per word row) of
// the rows [8t, 8t+8) of the step and writes 8 rows x 16 bytes, so the 8
// lanes of a row group store 128 contiguous bytes of one output row. The
// kernel is bound by the fp16 writes (2 bytes per weight against ~0.5 read).
#include "exq_device.cuh"
#include "exq_internal.h"

namespace exq {
namespace {

__device__ unsigned g_dequant_err;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct DequantArgs {
  const uint32_t* qweight;
  const uint16_t* scales;
  const uint32_t* q_scale;      // EXL2 two-level codes [S, N / 8]
  const uint16_t* q_scale_max;  // EXL2 two-level column maxima [N]
  const uint32_t* qzeros;
  const int32_t* perm;
  const uint32_t* seg_off;
  uint16_t* W;
  int K, N, n_steps, gs_steps, n_word_rows;
};

__device__ __forceinline__ uint4 ld_stream(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(uint16_t* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint32_t comp8(const uint4& a, const uint4& b, int c) {
  const uint4& v = c < 4 ? a : b;
  const int i = c & 3;
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// QS: two-level scales, s2 = the exact fractions (c + 1) / 16 and m2 the
// column maxima (the first multiply is exact, the second is the rounding)
template <int B, bool QS>
__device__ __forceinline__ void exl2_block(const uint4 (&wa)[2], const uint4 (&wb)[2], int off,
                                           const uint32_t (&s2)[8], const uint32_t (&m2)[8], uint32_t (&P)[8][4]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t a = comp8(wa[0], wa[1], c), b = comp8(wb[0], wb[1], c);
    unpack8<B>(fshr(a, b, off), b >> off, P[c]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      P[c][i] = hmul2(P[c][i], s2[c]);
      if constexpr (QS) P[c][i] = hmul2(P[c][i], m2[c]);
    }
  }
}

template <int FMT, bool PERM>
__global__ void __launch_bounds__(kThreads) dequant_kernel(const __grid_constant__ DequantArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int s = blockIdx.y * kWarps + warp;  // step (32 stored rows)
  const int col = blockIdx.x * 64 + 8 * g;
  if (s >= a.n_steps || col >= a.N) return;

  uint32_t P[8][4];
  uint32_t s2[8], m2[8];
  uint4 sv, mv;
  if constexpr (FMT == EXQ_FMT_GPTQ4) {
    const int grp = s / a.gs_steps;
    const uint4 w0 = ld_stream(a.qweight + static_cast<size_t>(4 * s + t) * a.N + col);
    const uint4 w1 = ld_stream(a.qweight + static_cast<size_t>(4 * s + t) * a.N + col + 4);
    sv = __ldg(reinterpret_cast<const uint4*>(a.scales + static_cast<size_t>(grp) * a.N + col));
    const uint32_t zw = __ldg(a.qzeros + static_cast<size_t>(grp) * (a.N >> 3) + (col >> 3));
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t zlo, zhi;
      gptq_zero_consts((zw >> (4 * c)) & 0xFu, zlo, zhi);
      const uint32_t h = comp8(sv, sv, c >> 1);
      s2[c] = (c & 1) ? prmt(h, h, 0x3232) : prmt(h, h, 0x1010);
      unpack8_gptq(comp8(w0, w1, c), zlo, zhi, P[c]);
#pragma unroll
      for (int i = 0; i < 4; ++i) P[c][i] = hmul2(P[c][i], s2[c]);
    }
  } else {
    const unsigned o0 = __ldg(a.seg_off + s), o1 = __ldg(a.seg_off + s + 1);
    const int b = static_cast<int>(o1 - o0);
    const bool ok = (b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8) && o1 > o0 &&
                    o1 <= static_cast<unsigned>(a.n_word_rows);
    int wi = 0, off = 0;
    if (ok) block_window(b, t, wi, off);
    const size_t row = static_cast<size_t>(o0) + wi;
    uint4 wa[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    uint4 wb[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (ok) {
      wa[0] = ld_stream(a.qweight + row * a.N + col);
      wa[1] = ld_stream(a.qweight + row * a.N + col + 4);
      if (block_needs_second(b, off)) {
        wb[0] = ld_stream(a.qweight + (row + 1) * a.N + col);
        wb[1] = ld_stream(a.qweight + (row + 1) * a.N + col + 4);
      }
    }
    if constexpr (FMT == EXQ_FMT_EXL2_QSCALE) {
      // the 8 columns' codes are one word (-> exact fractions); their maxima one 16-byte vector
      const uint32_t cw = __ldg(a.q_scale + static_cast<size_t>(s) * (a.N >> 3) + (col >> 3));
      mv = __ldg(reinterpret_cast<const uint4*>(a.q_scale_max + col));
      sv.x = two_level_frac2((cw & 0xFFu) | ((cw & 0xF0u) << 12));
      sv.y = two_level_frac2(((cw >> 8) & 0xFFu) | ((cw & 0xF000u) << 4));
      sv.z = two_level_frac2(((cw >> 16) & 0xFFu) | ((cw >> 4) & 0xF0000u));
      sv.w = two_level_frac2((cw >> 24) | ((cw >> 12) & 0xF0000u));
    } else {
      sv = __ldg(reinterpret_cast<const uint4*>(a.scales + static_cast<size_t>(s) * a.N + col));
      mv = sv;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t h = comp8(sv, sv, c >> 1), hm = comp8(mv, mv, c >> 1);
      s2[c] = (c & 1) ? prmt(h, h, 0x3232) : prmt(h, h, 0x1010);
      m2[c] = (c & 1) ? prmt(hm, hm, 0x3232) : prmt(hm, hm, 0x1010);
    }
    constexpr bool QS = FMT == EXQ_FMT_EXL2_QSCALE;
    switch (ok ? b : 0) {
      case 2: exl2_block<2, QS>(wa, wb, off, s2, m2, P); break;
      case 3: exl2_block<3, QS>(wa, wb, off, s2, m2, P); break;
      case 4: exl2_block<4, QS>(wa, wb, off, s2, m2, P); break;
      case 5: exl2_block<5, QS>(wa, wb, off, s2, m2, P); break;
      case 6: exl2_block<6, QS>(wa, wb, off, s2, m2, P); break;
      case 8: exl2_block<8, QS>(wa, wb, off, s2, m2, P); break;
      default:
        atomicOr(&g_dequant_err, kDevErrBadSegment);
#pragma unroll
        for (int c = 0; c < 8; ++c)
#pragma unroll
          for (int i = 0; i < 4; ++i) P[c][i] = 0u;
    }
  }

  // rows r = 8t + i (i < 4: low halves of P[.][i]; i >= 4: high halves of P[.][i-4])
  int dst[8];
  const int r0 = s * 32 + 8 * t;
  if constexpr (PERM) {
    const int4 p0 = __ldg(reinterpret_cast<const int4*>(a.perm + r0));
    const int4 p1 = __ldg(reinterpret_cast<const int4*>(a.perm + r0 + 4));
    dst[0] = p0.x; dst[1] = p0.y; dst[2] = p0.z; dst[3] = p0.w;
    dst[4] = p1.x; dst[5] = p1.y; dst[6] = p1.z; dst[7] = p1.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = r0 + i;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 lo, hi;
    lo.x = prmt(P[0][i], P[1][i], 0x5410);
    lo.y = prmt(P[2][i], P[3][i], 0x5410);
    lo.z = prmt(P[4][i], P[5][i], 0x5410);
    lo.w = prmt(P[6][i], P[7][i], 0x5410);
    hi.x = prmt(P[0][i], P[1][i], 0x7632);
    hi.y = prmt(P[2][i], P[3][i], 0x7632);
    hi.z = prmt(P[4][i], P[5][i], 0x7632);
    hi.w = prmt(P[6][i], P[7][i], 0x7632);
    st_stream(a.W + static_cast<size_t>(dst[i]) * a.N + col, lo);
    st_stream(a.W + static_cast<size_t>(dst[i + 4]) * a.N + col, hi);
  }
}

}  // namespace

exq_status launch_dequant(const exq_weight& w, uint16_t* W_out, cudaStream_t stream) {
  DequantArgs args{};
  args.qweight = w.qweight;
  args.scales = w.scales;
  args.q_scale = w.q_scale;
  args.q_scale_max = w.q_scale_max;
  args.qzeros = w.qzeros;
  args.perm = w.perm;
  args.seg_off = w.seg_word_off;
  args.W = W_out;
  args.K = w.K;
  args.N = w.N;
  args.n_steps = w.K / 32;
  args.gs_steps = w.format == EXQ_FMT_GPTQ4 ? w.group_size / 32 : 1;
  args.n_word_rows = w.n_word_rows;
  const dim3 grid((w.N + 63) / 64, (args.n_steps + kWarps - 1) / kWarps, 1);
  const bool perm = w.perm != nullptr;
  if (w.format == EXQ_FMT_GPTQ4) {
    if (perm) dequant_kernel<EXQ_FMT_GPTQ4, true><<<grid, kThreads, 0, stream>>>(args);
    else dequant_kernel<EXQ_FMT_GPTQ4, false><<<grid, kThreads, 0, stream>>>(args);
  } else if (w.format == EXQ_FMT_EXL2) {
    if (perm) dequant_kernel<EXQ_FMT_EXL2, true><<<grid, kThreads, 0, stream>>>(args);
    else dequant_kernel<EXQ_FMT_EXL2, false><<<grid, kThreads, 0, stream>>>(args);
  } else {
    if (perm) dequant_kernel<EXQ_FMT_EXL2_QSCALE, true><<<grid, kThreads, 0, stream>>>(args);
    else dequant_kernel<EXQ_FMT_EXL2_QSCALE, false><<<grid, kThreads, 0, stream>>>(args);
  }
  if (cudaGetLastError() != cudaSuccess) return EXQ_ERR_CUDA;
  return EXQ_OK;
}

unsigned take_dequant_errors(cudaStream_t stream) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_dequant_err, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return ~0u;
  if (cudaMemcpyToSymbolAsync(g_dequant_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
      cudaSuccess)
    return ~0u;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
  return v;
}

}  // namespace exq
