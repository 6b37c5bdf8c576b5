// Quantized KV cache codec, Q4 / Q6 / Q8.
//
// The ExLlamaV2 blog post ("ExLlamaV2: The fastest inference engine for
// quantized Llama/HF models") lists a Q4 / Q6 / Q8 KV cache (comparison table;
// "Step 2: Use the right cache mode for your context length") and costs it
// at half a byte (Q4) and one byte (Q8) per cached element ("Production
// Considerations", VRAM estimate); the codec itself is not described. This
// one: a group is the D values of one (token, head); symmetric with
// qmax = 2^(b-1) - 1;
//   s = fp16_RN(fp32_RN(amax / qmax)),
//   q = clamp(rint(fp32_RN(x / s)), -qmax - 1, qmax)  (0 where s = 0),
//   u = q + 2^(b-1), code i of the group at bits [i b, i b + b) of its
//   little-endian word stream;
// read back as fp16_RN((u - 2^(b-1)) s). Every integer decision is an IEEE
// fp32 division rounded to nearest even, then round-half-even to an integer.
//
// Both kernels are bound by HBM. A warp handles four groups, lane l holding
// the D / 32 consecutive values [l D/32, (l+1) D/32) of each, so a group moves
// as one contiguous block (D * 2 bytes of fp16, D * b / 8 bytes of codes); all
// of a warp's loads are issued before any of its arithmetic, to keep enough
// bytes in flight per SM.
#include <type_traits>

#include "exq_device.cuh"
#include "exq_internal.h"

namespace exq {
namespace {

constexpr int kWarps = 8;  // groups per 256-thread block

// x / C rounded to nearest even in fp32, for x an fp16 magnitude (amax) and
// C = qmax in {7, 31, 127}: the quotient x y with y = RN(1 / C), corrected by
// one fma with its remainder (the division-by-a-constant method of Cornea,
// Harrison and Tang, "Scientific Computing on Itanium-based Systems", FMA
// correction step). For these C every positive finite fp16 x gives the
// correctly rounded quotient, checked exhaustively against exact rational
// rounding in tests/test_kv_division.py; three instructions instead of a
// full IEEE division.
template <int C>
__device__ __forceinline__ float div_by_const(float x) {
  // RN(1 / C), written out so that it does not depend on constant folding
  constexpr float y = C == 7 ? 0x1.24924ap-3f : C == 31 ? 0x1.084210p-5f : 0x1.020408p-7f;
  const float q = __fmul_rn(x, y);
  const float r = __fmaf_rn(-q, static_cast<float>(C), x);
  return __fmaf_rn(r, y, q);
}

// 1 / s from the hardware's approximate reciprocal (PTX `rcp.approx.ftz.f32`,
// at most 1 ulp from 1 / s over the whole range; s is an fp16 value, so
// never an fp32 subnormal). x * inv is then within |x / s| 2^-22 of
// fp32_RN(x / s): 2^-15 for the codes that are not clamped (|x / s| <=
// 128), half the window below in which the exact quotient decides.
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

template <int VPL>  // values per lane: D / 32
struct Vec;
template <>
struct Vec<2> {
  using T = uint32_t;
};
template <>
struct Vec<4> {
  using T = uint2;
};
template <>
struct Vec<8> {
  using T = uint4;
};

template <int VPL>
__device__ __forceinline__ void unpack_halves(const typename Vec<VPL>::T& v, uint32_t (&h)[VPL]) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
  for (int i = 0; i < VPL / 2; ++i) {
    h[2 * i] = w[i] & 0xFFFFu;
    h[2 * i + 1] = w[i] >> 16;
  }
}

constexpr int gcd32(int c) { return c % 32 == 0 ? 32 : c % 16 == 0 ? 16 : c % 8 == 0 ? 8 : 4; }

// The group's code words from the lanes' bit chunks (lane l holds stream bits
// [l C, l C + C), C = kChunk <= 64): word w gathers, by warp shuffles, the at
// most NC chunks that overlap bits [32 w, 32 w + 32). Every lane calls it.
template <int kChunk, int kWords>
__device__ __forceinline__ void store_words(unsigned long long chunk, uint32_t* __restrict__ dst, int lane) {
  if constexpr (kChunk == 64) {  // two whole words per lane
    *reinterpret_cast<uint2*>(dst + 2 * lane) =
        make_uint2(static_cast<uint32_t>(chunk), static_cast<uint32_t>(chunk >> 32));
    return;
  } else if constexpr (kChunk == 32) {  // one whole word per lane
    dst[lane] = static_cast<uint32_t>(chunk);
    return;
  } else if constexpr (kChunk == 24) {  // four lanes fill three words: lane 4k + i (i < 3) writes word 3k + i
    const uint32_t c = static_cast<uint32_t>(chunk);
    const uint32_t next = __shfl_down_sync(0xffffffffu, c, 1);
    const int i = lane & 3;
    if (i < 3) dst[3 * (lane >> 2) + i] = (c >> (8 * i)) | (next << (24 - 8 * i));
    return;
  } else if constexpr (kChunk == 16 || kChunk == 8) {  // 32 / kChunk lanes fill a word
    constexpr int kPer = 32 / kChunk;
    uint32_t word = static_cast<uint32_t>(chunk);
#pragma unroll
    for (int i = 1; i < kPer; ++i)
      word |= __shfl_down_sync(0xffffffffu, static_cast<uint32_t>(chunk), i) << (i * kChunk);
    if (lane % kPer == 0) dst[lane / kPer] = word;
    return;
  }
  constexpr int NC = (kChunk - gcd32(kChunk) + 32 + kChunk - 1) / kChunk;
#pragma unroll
  for (int r = 0; r < (kWords + 31) / 32; ++r) {
    const int w = 32 * r + lane;
    const int l0 = min(32 * w / kChunk, 31);
    const int sh = 32 * w - l0 * kChunk;  // the word's first bit inside chunk l0
    uint32_t word = 0;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int src = min(l0 + c, 31);
      unsigned long long v;
      if constexpr (kChunk <= 32) {
        v = __shfl_sync(0xffffffffu, static_cast<uint32_t>(chunk), src);
      } else {
        const uint32_t lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(chunk), src);
        const uint32_t hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(chunk >> 32), src);
        v = (static_cast<unsigned long long>(hi) << 32) | lo;
      }
      const int pos = c * kChunk - sh;  // chunk l0 + c starts this many bits into the word
      if (l0 + c <= 31 && pos < 32) word |= pos >= 0 ? static_cast<uint32_t>(v << pos) : static_cast<uint32_t>(v >> -pos);
    }
    if (w < kWords) dst[w] = word;
  }
}

template <int VPL, int B, int GPW>
__global__ void __launch_bounds__(kWarps * 32)
    kv_quantize_kernel(const uint16_t* __restrict__ x, long long n_groups, uint32_t* __restrict__ codes,
                       uint16_t* __restrict__ scales) {
  constexpr int D = 32 * VPL;
  constexpr int kWords = D * B / 32;   // words of a group
  constexpr int kChunk = VPL * B;      // bits of one lane (8..64)
  constexpr int kQmax = (1 << (B - 1)) - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the block's groups: k * kWarps + warp, k < GPW (each k a contiguous run of kWarps groups)
  const long long g0 = static_cast<long long>(blockIdx.x) * kWarps * GPW + warp;

  using V = typename Vec<VPL>::T;
  V raw[GPW];
#pragma unroll
  for (int k = 0; k < GPW; ++k) {  // every load of the warp first
    const long long g = g0 + k * kWarps;
    if (g < n_groups) raw[k] = *reinterpret_cast<const V*>(x + g * D + lane * VPL);
  }

#pragma unroll
  for (int k = 0; k < GPW; ++k) {
    const long long g = g0 + k * kWarps;
    if (g >= n_groups) break;  // warp-uniform
    uint32_t h[VPL];
    unpack_halves<VPL>(raw[k], h);
    float xf[VPL];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      xf[i] = __half2float(__ushort_as_half(static_cast<unsigned short>(h[i])));
      amax = fmaxf(amax, fabsf(xf[i]));
    }
    // non-negative floats order as their bit patterns
    amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
    static_assert(kQmax == 7 || kQmax == 31 || kQmax == 127, "div_by_const is checked for these only");
    const __half s16 = __float2half_rn(div_by_const<kQmax>(amax));
    const float s = __half2float(s16);
    const float inv = s != 0.f ? rcp_approx(s) : 0.f;  // s = 0: every q is 0

    // q = rint(fp32_RN(x / s)): from x * inv, except where that lies within
    // 2^-14 of a half-integer; one test per lane for its VPL values
    int q[VPL];
    bool near_tie = false;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      const float r = xf[i] * inv;
      q[i] = __float2int_rn(r);
      near_tie |= fabsf(r - static_cast<float>(q[i])) > 0.5f - 0x1p-14f;
    }
    if (near_tie)
#pragma unroll
      for (int i = 0; i < VPL; ++i) q[i] = __float2int_rn(__fdiv_rn(xf[i], s));
    // A normal fp16 s is within 2^-11 (plus the fp32 quotient's 2^-24) of
    // amax / qmax, so |x / s| < qmax (1 + 2^-10) < qmax + 1/2 and every q is
    // already in range; only a subnormal s (amax < 2^-14 qmax), with fewer
    // significant bits, needs the clamp. The test is the same for the whole
    // warp (s is the group's).
    if (s < 0x1p-14f)
#pragma unroll
      for (int i = 0; i < VPL; ++i) q[i] = max(-kQmax - 1, min(kQmax, q[i]));
    using Chunk = std::conditional_t<(kChunk <= 32), uint32_t, unsigned long long>;
    Chunk chunk = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) chunk |= static_cast<Chunk>(q[i] + (1 << (B - 1))) << (i * B);
    store_words<kChunk, kWords>(chunk, codes + g * kWords, lane);
    if (lane == 0) scales[g] = __half_as_ushort(s16);
  }
}

template <int VPL, int B, int GPW>
__global__ void __launch_bounds__(kWarps * 32)
    kv_dequantize_kernel(const uint32_t* __restrict__ codes, const uint16_t* __restrict__ scales, long long n_groups,
                         uint16_t* __restrict__ x_out) {
  constexpr int D = 32 * VPL;
  constexpr int kWords = D * B / 32;
  constexpr int kChunk = VPL * B;
  constexpr uint32_t kMask = (1u << B) - 1u;
  constexpr int kZ = 1 << (B - 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long g0 = static_cast<long long>(blockIdx.x) * kWarps * GPW + warp;
  const int off = lane * kChunk;
  constexpr bool kTwo = (kChunk & 31) != 0 || kChunk > 32;  // some lane's bits cross a word boundary

  uint32_t lo[GPW], hi[GPW], sc[GPW];
#pragma unroll
  for (int k = 0; k < GPW; ++k) {  // every load of the warp first
    const long long g = g0 + k * kWarps;
    lo[k] = hi[k] = sc[k] = 0u;
    if (g < n_groups) {
      const uint32_t* gw = codes + g * kWords;
      lo[k] = __ldg(gw + (off >> 5));
      if (kTwo && (off & 31) + kChunk > 32) hi[k] = __ldg(gw + (off >> 5) + 1);  // inside the group
      sc[k] = __ldg(scales + g);
    }
  }
  // (u - z) exactly in fp16: u planted in the mantissa of 1024, then - (1024 + z)
  constexpr uint32_t bias = pack2(f16_bits(-(1024 + kZ)), f16_bits(-(1024 + kZ)));
#pragma unroll
  for (int k = 0; k < GPW; ++k) {
    const long long g = g0 + k * kWarps;
    if (g >= n_groups) break;
    const unsigned long long win = ((static_cast<unsigned long long>(hi[k]) << 32) | lo[k]) >> (off & 31);
    const uint32_t s2 = sc[k] | (sc[k] << 16);
    uint32_t out[VPL / 2];
#pragma unroll
    for (int i = 0; i < VPL / 2; ++i) {
      const uint32_t u0 = static_cast<uint32_t>(win >> (2 * i * B)) & kMask;
      const uint32_t u1 = static_cast<uint32_t>(win >> ((2 * i + 1) * B)) & kMask;
      out[i] = hmul2(hadd2(u0 | (u1 << 16) | kMagic, bias), s2);
    }
    using V = typename Vec<VPL>::T;
    *reinterpret_cast<V*>(x_out + g * D + lane * VPL) = *reinterpret_cast<const V*>(out);
  }
}

constexpr int kGpw = 4;  // groups per warp

using QuantFn = void (*)(const uint16_t*, long long, uint32_t*, uint16_t*);
using DequantFn = void (*)(const uint32_t*, const uint16_t*, long long, uint16_t*);

template <int VPL>
QuantFn quant_for_bits(int b) {
  return b == 4 ? kv_quantize_kernel<VPL, 4, kGpw>
                : b == 6 ? kv_quantize_kernel<VPL, 6, kGpw> : kv_quantize_kernel<VPL, 8, kGpw>;
}
template <int VPL>
DequantFn dequant_for_bits(int b) {
  return b == 4 ? kv_dequantize_kernel<VPL, 4, kGpw>
                : b == 6 ? kv_dequantize_kernel<VPL, 6, kGpw> : kv_dequantize_kernel<VPL, 8, kGpw>;
}

dim3 grid_for(long long n_groups) {
  return dim3(static_cast<unsigned>((n_groups + kWarps * kGpw - 1) / (kWarps * kGpw)));
}

}  // namespace

exq_status launch_kv_quantize(const uint16_t* x, long long n_groups, int D, int b, uint32_t* codes,
                              uint16_t* scales, cudaStream_t stream) {
  if (n_groups == 0) return EXQ_OK;
  const QuantFn fn = D == 64 ? quant_for_bits<2>(b) : D == 128 ? quant_for_bits<4>(b) : quant_for_bits<8>(b);
  fn<<<grid_for(n_groups), kWarps * 32, 0, stream>>>(x, n_groups, codes, scales);
  return cudaGetLastError() == cudaSuccess ? EXQ_OK : EXQ_ERR_CUDA;
}

exq_status launch_kv_dequantize(const uint32_t* codes, const uint16_t* scales, long long n_groups, int D, int b,
                                uint16_t* x_out, cudaStream_t stream) {
  if (n_groups == 0) return EXQ_OK;
  const DequantFn fn =
      D == 64 ? dequant_for_bits<2>(b) : D == 128 ? dequant_for_bits<4>(b) : dequant_for_bits<8>(b);
  fn<<<grid_for(n_groups), kWarps * 32, 0, stream>>>(codes, scales, n_groups, x_out);
  return cudaGetLastError() == cudaSuccess ? EXQ_OK : EXQ_ERR_CUDA;
}

}  // namespace exq
