// Device helpers shared by the libexq kernels: fp16x2 arithmetic on raw bit
// patterns and the per-width code unpackers.
//
// Unpacking follows the ExLlamaV2 blog post ("ExLlamaV2: The fastest
// inference engine for quantized Llama/HF models", section "How the Fused CUDA
// Kernel Works"): a code is a bit field of a packed uint32, dequantised as
// (code - zero) * scale. Here the subtraction is done exactly in fp16 by
// planting the code in the mantissa of 1024.0 (0x6400 | code == 1024 + code),
// so that w = fp16_RN((q - z) * s) takes exactly one rounding, in the final
// fp16 multiply.
//
// Every unpacker produces, for the 8 consecutive codes v0..v7 of one thread's
// block, four fp16x2 words P[i] = (v_i - z, v_{i+4} - z), i = 0..3 (low half
// first). Consumers arrange the matching activations in the same order.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace exq {

// ---------------------------------------------------------------- bit ops

// (a & mask) | set
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t set) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(set));
  return r;
}

// (a & m) | (b & ~m)
__device__ __forceinline__ uint32_t bitselect(uint32_t a, uint32_t b, uint32_t m) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xE4;" : "=r"(r) : "r"(a), "r"(b), "r"(m));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  return __byte_perm(a, b, sel);
}

// low 32 bits of (hi:lo) >> s, 0 <= s < 32
__device__ __forceinline__ uint32_t fshr(uint32_t lo, uint32_t hi, uint32_t s) {
  return __funnelshift_r(lo, hi, s);
}

// ---------------------------------------------------------------- fp16x2 on bit patterns

__device__ __forceinline__ uint32_t hadd2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Bit pattern of an fp16 value that is +-(integer < 2048) or +-2^-p; exact.
__host__ __device__ constexpr uint32_t f16_bits(int v) {
  // integers only: |v| < 2048
  return v == 0 ? 0u
                : ((v < 0 ? 0x8000u : 0u) |
                   [](unsigned a) constexpr {
                     int e = 0;
                     while ((a >> e) > 1) ++e;                   // leading bit
                     const unsigned frac = (a << (10 - e)) & 0x3FFu;  // exact for e <= 10
                     return static_cast<uint32_t>(((e + 15) << 10) | frac);
                   }(static_cast<unsigned>(v < 0 ? -v : v)));
}

__host__ __device__ constexpr uint32_t f16_pow2_neg(int p) {  // 2^-p, 0 <= p <= 14
  return static_cast<uint32_t>((15 - p) << 10);
}

__host__ __device__ constexpr uint32_t pack2(uint32_t lo, uint32_t hi) { return lo | (hi << 16); }

static_assert(f16_bits(1024) == 0x6400, "f16 1024");
static_assert(f16_bits(-1026) == 0xE402, "f16 -1026");
static_assert(f16_bits(258) == 0x5C08, "f16 258");
static_assert(f16_pow2_neg(4) == 0x2C00, "f16 1/16");

constexpr uint32_t kMagic = 0x64006400u;  // (1024.0, 1024.0)

// v = (1024 + 2^plo * a, 1024 + 2^phi * b) with a, b in the mantissa at bit
// offsets plo / phi; returns (a - z, b - z) exactly.
template <int PLO, int PHI, int Z>
__device__ __forceinline__ uint32_t unbias(uint32_t v) {
  if constexpr (PLO == 0 && PHI == 0) {
    return hadd2(v, pack2(f16_bits(-(1024 + Z)), f16_bits(-(1024 + Z))));
  } else {
    constexpr uint32_t mul = pack2(f16_pow2_neg(PLO), f16_pow2_neg(PHI));
    constexpr uint32_t add = pack2(f16_bits(-((1024 >> PLO) + Z)), f16_bits(-((1024 >> PHI) + Z)));
    return hfma2(v, mul, add);
  }
}

// ---------------------------------------------------------------- unpackers
// Window (lo, hi): 64 bits whose bit 0 is the first code of the block.

// EXL2, width B, zero 2^(B-1).
template <int B>
__device__ __forceinline__ void unpack8(uint32_t lo, uint32_t hi, uint32_t (&P)[4]) {
  constexpr int Z = 1 << (B - 1);
  if constexpr (B == 2) {
    // codes 0..3 in byte 0, 4..7 in byte 1: move byte 1 to byte 2
    const uint32_t u = prmt(lo, lo, 0x1110);
    P[0] = unbias<0, 0, Z>(and_or(u, 0x00030003u, kMagic));
    P[1] = unbias<2, 2, Z>(and_or(u, 0x000C000Cu, kMagic));
    P[2] = unbias<4, 4, Z>(and_or(u, 0x00300030u, kMagic));
    P[3] = unbias<6, 6, Z>(and_or(u, 0x00C000C0u, kMagic));
  } else if constexpr (B == 3) {
    // codes 4..7 (bits 12..23) moved up by 4 -> code i+4 sits 16 bits above code i
    const uint32_t u = bitselect(lo, lo << 4, 0x00000FFFu);
    const uint32_t u6 = u >> 6;
    P[0] = unbias<0, 0, Z>(and_or(u, 0x00070007u, kMagic));
    P[1] = unbias<3, 3, Z>(and_or(u, 0x00380038u, kMagic));
    P[2] = unbias<6, 6, Z>(and_or(u, 0x01C001C0u, kMagic));
    P[3] = unbias<3, 3, Z>(and_or(u6, 0x00380038u, kMagic));
  } else if constexpr (B == 4) {
    const uint32_t u8 = lo >> 8;
    P[0] = unbias<0, 0, Z>(and_or(lo, 0x000F000Fu, kMagic));
    P[1] = unbias<4, 4, Z>(and_or(lo, 0x00F000F0u, kMagic));
    P[2] = unbias<0, 0, Z>(and_or(u8, 0x000F000Fu, kMagic));
    P[3] = unbias<4, 4, Z>(and_or(u8, 0x00F000F0u, kMagic));
  } else if constexpr (B == 5) {
    // window >> 5i: code i at bit 0, code i+4 at bit 20 (= offset 4 in the high half)
    P[0] = unbias<0, 4, Z>(and_or(lo, 0x01F0001Fu, kMagic));
    P[1] = unbias<0, 4, Z>(and_or(fshr(lo, hi, 5), 0x01F0001Fu, kMagic));
    P[2] = unbias<0, 4, Z>(and_or(fshr(lo, hi, 10), 0x01F0001Fu, kMagic));
    P[3] = unbias<0, 4, Z>(and_or(fshr(lo, hi, 15), 0x01F0001Fu, kMagic));
  } else if constexpr (B == 6) {
    const uint32_t w4 = fshr(lo, hi, 4);
    P[0] = unbias<0, 0, Z>(and_or(prmt(lo, hi, 0x3300), 0x003F003Fu, kMagic));  // bytes 0 | 3
    P[1] = unbias<2, 2, Z>(and_or(prmt(w4, w4, 0x3300), 0x00FC00FCu, kMagic));
    P[2] = unbias<4, 4, Z>(and_or(prmt(lo, hi, 0x5421), 0x03F003F0u, kMagic));  // bits 8.. | 32..
    P[3] = unbias<2, 2, Z>(and_or(prmt(lo, hi, 0x6532), 0x00FC00FCu, kMagic));  // bits 16.. | 40..
  } else {  // B == 8: codes 0..3 = bytes of lo, 4..7 = bytes of hi
    static_assert(B == 8, "width");
    P[0] = unbias<0, 0, Z>(and_or(prmt(lo, hi, 0x4400), 0x00FF00FFu, kMagic));
    P[1] = unbias<0, 0, Z>(and_or(prmt(lo, hi, 0x5511), 0x00FF00FFu, kMagic));
    P[2] = unbias<0, 0, Z>(and_or(prmt(lo, hi, 0x6622), 0x00FF00FFu, kMagic));
    P[3] = unbias<0, 0, Z>(and_or(prmt(lo, hi, 0x7733), 0x00FF00FFu, kMagic));
  }
}

// GPTQ 4-bit with a per-column runtime zero z:
//   zlo = (-(1024 + z), -(1024 + z)), zhi = (-(64 + z), -(64 + z)).
__device__ __forceinline__ void unpack8_gptq(uint32_t w, uint32_t zlo, uint32_t zhi, uint32_t (&P)[4]) {
  constexpr uint32_t sixteenth = pack2(f16_pow2_neg(4), f16_pow2_neg(4));
  const uint32_t w8 = w >> 8;
  P[0] = hadd2(and_or(w, 0x000F000Fu, kMagic), zlo);
  P[1] = hfma2(and_or(w, 0x00F000F0u, kMagic), sixteenth, zhi);
  P[2] = hadd2(and_or(w8, 0x000F000Fu, kMagic), zlo);
  P[3] = hfma2(and_or(w8, 0x00F000F0u, kMagic), sixteenth, zhi);
}

// zero nibble z (0..15) -> (zlo, zhi) constants for unpack8_gptq
__device__ __forceinline__ void gptq_zero_consts(uint32_t z, uint32_t& zlo, uint32_t& zhi) {
  const uint32_t zz = z | (z << 16);
  zlo = zz | 0xE400E400u;          // -(1024 + z): sign | exponent of 1024 | z in the mantissa
  zhi = (zz << 4) | 0xD400D400u;   // -(64 + z):   sign | exponent of 64   | 16 z (mantissa step 1/16)
}

// EXL2 two-level scales, two columns at once: the codes c_lo and c_hi sit in
// bits 0..3 and 16..19 of cc (other bits are ignored). Returns the exact
// fractions ((c_lo + 1) / 16, (c_hi + 1) / 16): (1024 + c) / 16 - 1023 / 16
// comes out exact from one fp16 fma. The weight is then
// fp16_RN(fp16_RN((q - z) * f) * m): the inner product (q - z) (c + 1) / 16
// has at most 7 + 4 significant bits and lies in [1/16, 128] (or is 0), so it
// is exact, and the multiply by the column maximum m is the one rounding of
// w = fp16_RN((q - z) * ((c + 1) / 16) * m).
constexpr uint32_t kNeg1023Over16 = f16_bits(-1023) - (4u << 10);  // -63.9375: exponent lowered by 4
static_assert(kNeg1023Over16 == 0xD3FE, "f16 -1023/16");

__device__ __forceinline__ uint32_t two_level_frac2(uint32_t cc) {
  constexpr uint32_t sixteenth = pack2(f16_pow2_neg(4), f16_pow2_neg(4));
  constexpr uint32_t bias = pack2(kNeg1023Over16, kNeg1023Over16);
  return hfma2(and_or(cc, 0x000F000Fu, kMagic), sixteenth, bias);
}

// x / s rounded to an integer as rint(fp32_RN(x / s)): the quotient comes
// from a multiply by fp32_RN(1 / s), which is within 3 * 2^-24 |x / s| of the
// correctly rounded one; only where that leaves the quotient within 2^-14 of
// a half-integer (|x / s| <= 256: 4.6e-5 < 2^-14) does the exact division
// decide. Beyond 256 the code is clamped whichever quotient is used.
__device__ __forceinline__ int round_quotient(float x, float s, float inv) {
  float r = x * inv;
  if (fabsf(fabsf(r - rintf(r)) - 0.5f) < 0x1p-14f) r = __fdiv_rn(x, s);
  return __float2int_rn(r);
}

// Bit-window of one 8-code block: block t (0..3) of a segment of width b
// starts at stream bit 8 t b. Returns the first word row (relative to the
// segment) and the bit offset inside it.
__device__ __forceinline__ void block_window(int b, int t, int& word, int& off) {
  const int bit = 8 * t * b;
  word = bit >> 5;
  off = bit & 31;
}

// does block t of a width-b segment spill into a second word?
__device__ __forceinline__ bool block_needs_second(int b, int off) { return off + 8 * b > 32; }

// fp16x2 of a scalar fp16 in both halves
__device__ __forceinline__ uint32_t splat(uint32_t h16) { return prmt(h16, h16, 0x1010); }

}  // namespace exq
