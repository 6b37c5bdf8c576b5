// Decode-sized fused quantized matmul, 1 <= M <= 16:  y = x . dequant(Wq).
//
// Follows the fused kernel of the ExLlamaV2 blog post ("ExLlamaV2: The fastest
// inference engine for quantized Llama/HF models", section "How the Fused CUDA
// Kernel Works"): the packed weights stream from memory once, codes are
// unpacked in registers, multiplied into fp32 sums and the result is written
// as fp16. The act-order row remapping (ExLlamaV2 README, "EXL2
// quantization") is applied to x (gathered into stored-row order), so the
// weights stream in stored order.
//
// GB300 mapping:
//  * Work is the set of (256-column tile, 32-row step) pairs, ordered by K
//    chunk (a chunk is as many steps as the staged activations fit in shared
//    memory), then tile, then step. Every CTA (one per SM) takes an equal
//    contiguous share, so all SMs stream the same number of bytes whatever N
//    and K are. A share falls into pieces, one per tile it touches.
//  * Inside a piece the warps form 4 column groups (64 columns each) x KG K
//    groups; a K group owns a contiguous run of the piece's steps, and the 4
//    warps of a K group read the same word rows side by side (1 KB per row).
//  * Per step a lane (g = lane / 4, t = lane % 4) owns 8 columns (4g .. 4g+3
//    and 32+4g .. 32+4g+3 of its group) of the 8-row block t of the step: the
//    8 lanes of a word row read whole 128-byte lines. Its word rows and scales
//    travel by cp.async into a private slot of a P-stage shared-memory ring,
//    so P - 1 steps of every lane are in flight while it works on the current
//    one, with no cross-warp hand-shake; the fetches run ahead across piece
//    boundaries.
//  * Codes are planted in the mantissa of 1024 (0x6400 | code << p), the zero
//    is taken off exactly in fp16 and each pair is scaled once
//    (w = fp16_RN((q - z) s), the definition), then fed to mma.sync m16n8k16
//    (fp16 in, fp32 accumulate) as the A operand of a swapped product
//    (A = W^T, B = x^T). The K order inside a 16-slab is free as long as A and
//    B agree, so x is staged in the pair order the unpackers produce.
//  * At the end of a piece the K groups' partial sums are added in shared
//    memory in K-group order. A tile that one CTA covers whole is written to
//    y; the pieces of a shared tile go to the caller's workspace and the CTA
//    that arrives last (one atomic counter per tile) adds them in piece order,
//    writes y and puts the counter back to zero. Deterministic, and no CTA
//    ever waits on another.
//  * An act-order layer's x is gathered into stored-row order by a small
//    kernel first (into the workspace), once per call rather than once per
//    CTA.
//  * Programmatic dependent launch: the kernels let the next launch start
//    early; the GEMV starts fetching weights before it waits for the previous
//    kernel; x, y and the workspace are touched only after that wait.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "exq_device.cuh"
#include "exq_internal.h"

namespace exq {
namespace {

__device__ unsigned g_gemv_err;

constexpr int kTN = 256;                     // columns per tile
constexpr int kCG = 4;                       // 64-column groups of a tile, one per warp of a K group
constexpr int kCounterBytes = 64 * 1024;     // workspace counter region (zero between calls)
constexpr int kP = 4;                        // pipeline stages per lane
constexpr int kSlotBytes = 80;               // per lane and stage: a0 a1 | b0 b1 | scales

// Launch shapes: M <= 8 with 16 warps (4 column groups x 4 K groups); M <= 16
// (two 8-token blocks) with 8 (4 x 2).
__host__ __device__ constexpr int mode_for(int M) { return M <= 8 ? 0 : 1; }
__host__ __device__ constexpr int warps_of(int mode) { return mode == 0 ? 16 : 8; }

struct GemvArgs {
  const uint32_t* qweight;
  const uint16_t* scales;
  const uint32_t* qzeros;
  const uint32_t* seg_off;
  const uint16_t* x;
  uint16_t* y;
  uint32_t* counters;   // [n_tiles], zero between calls
  float* partials;      // [n_tiles][max_pieces][M][kTN]
  int K, N, M;
  int n_steps;          // K / 32
  int gs_steps;         // GPTQ: group_size / 32; EXL2: 1
  int n_word_rows;
  int n_tiles;          // ceil(N / kTN)
  int kc_steps;         // steps per K chunk
  int n_chunks;
  int max_pieces;
  int xs_stride;        // halves per staged x row
  int total;            // n_tiles * n_steps
  // byte offsets in dynamic shared memory (from a 1024-aligned base)
  int off_flags, off_x, off_meta, off_red;
};

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// barrier of all NW warps of the CTA (id 1; __syncthreads uses 0)
template <int NW>
__device__ __forceinline__ void cta_barrier() {
  asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// 16-, 8- and 4-byte asynchronous global -> shared copies, one per thread,
// tracked per thread in commit groups
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- work split
// The work is the list of (chunk, tile, step) positions in that order
// (total < 2^31, checked on the host); CTA c owns [c * total / G,
// (c + 1) * total / G).

struct Split {
  int total, G, n_tiles, n_steps, kc_steps, n_chunks;

  __host__ __device__ int begin(int c) const {
    return static_cast<int>(static_cast<long long>(c) * total / G);
  }
  // the CTA that owns position p
  __host__ __device__ int owner(int p) const {
    return static_cast<int>((static_cast<long long>(p + 1) * G - 1) / total);
  }
  __host__ __device__ int chunk_len(int kc) const {
    return kc == n_chunks - 1 ? n_steps - kc * kc_steps : kc_steps;
  }
  __host__ __device__ int unit_begin(int kc, int tile) const {
    return kc * n_tiles * kc_steps + tile * chunk_len(kc);
  }
  // CTAs sharing unit (kc, tile) and the first of them
  __host__ __device__ int unit_pieces(int kc, int tile, int& first) const {
    const int u0 = unit_begin(kc, tile);
    first = owner(u0);
    return owner(u0 + chunk_len(kc) - 1) - first + 1;
  }
};

struct Piece {
  int kc, tile;
  int sa, sb;     // absolute steps [sa, sb)
  int slot, P;    // index among the tile's pieces, number of pieces
};

// the piece that starts at position p (< end) of CTA c's share
__device__ __forceinline__ Piece piece_at(const Split& sp, int c, int p, int end, int& next) {
  Piece pc;
  const int per_chunk = sp.n_tiles * sp.kc_steps;
  pc.kc = min(p / per_chunk, sp.n_chunks - 1);
  const int base = pc.kc * per_chunk;
  const int len = sp.chunk_len(pc.kc);
  const int rem = p - base;
  pc.tile = rem / len;
  const int sin = rem - pc.tile * len;
  next = min(end, base + (pc.tile + 1) * len);
  pc.sa = pc.kc * sp.kc_steps + sin;
  pc.sb = pc.sa + (next - p);
  pc.P = 0;
  pc.slot = 0;
  for (int k = 0; k < sp.n_chunks; ++k) {
    int first;
    const int n = sp.unit_pieces(k, pc.tile, first);
    if (k < pc.kc) pc.slot += n;
    if (k == pc.kc) pc.slot += c - first;
    pc.P += n;
  }
  return pc;
}

// steps [ws, we) of warp w (of NW) inside a piece
template <int NW>
__device__ __forceinline__ void warp_range(const Piece& pc, int w, int& ws, int& we) {
  const int len = pc.sb - pc.sa;
  const int L = (len + NW - 1) / NW;
  ws = min(pc.sb, pc.sa + w * L);
  we = min(pc.sb, ws + L);
}

// ---------------------------------------------------------------- one 32-row step
// Lane column c (0..7) is column 4g + c (c < 4) or 32 + 4g + c - 4 of the
// warp's 64-column group.

__device__ __forceinline__ int group_col(int c, int g) { return (c < 4 ? 0 : 28) + 4 * g + c; }

template <int MT>
__device__ __forceinline__ void zero_acc(float (&a)[MT][4][4]) {
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) a[mt][nt][i] = 0.f;
}

template <int MT>
__device__ __forceinline__ void mma_pair(float (&acc)[MT][4][4], int nt, const uint32_t (&P0)[4],
                                         const uint32_t (&P1)[4], const uint4& xb0, const uint4& xb1) {
  // A rows g / g + 8 = half columns 2nt / 2nt + 1; slab 0 takes pairs
  // 0 (k 2t, 2t+1) and 1 (k 2t+8, 2t+9), slab 1 pairs 2 and 3
  mma16816(acc[0][nt], P0[0], P1[0], P0[1], P1[1], xb0.x, xb0.y);
  mma16816(acc[0][nt], P0[2], P1[2], P0[3], P1[3], xb0.z, xb0.w);
  if constexpr (MT == 2) {
    mma16816(acc[1][nt], P0[0], P1[0], P0[1], P1[1], xb1.x, xb1.y);
    mma16816(acc[1][nt], P0[2], P1[2], P0[3], P1[3], xb1.z, xb1.w);
  }
}

// (s, s) of half column c from the half's 8 scales in v
__device__ __forceinline__ uint32_t scale_x2(const uint4& v, int c) {
  const uint32_t h = comp(v, c >> 1);
  return (c & 1) ? prmt(h, h, 0x3232) : prmt(h, h, 0x1010);
}

// EXL2 half step of width B: A = the word row of the lane's block (chunks
// 2hf, 2hf + 1), Bn = the next word row when the block spills over
template <int B, int MT>
__device__ __forceinline__ void exl2_half(const uint4& A0, const uint4& A1, const uint4& B0, const uint4& B1,
                                          const uint4& sc, uint32_t off, const uint4& xb0, const uint4& xb1,
                                          float (&acc)[MT][4][4]) {
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    uint32_t P[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 2 * nt + h;
      const uint32_t wa = comp(c < 4 ? A0 : A1, c & 3);
      uint32_t lo = wa, hi = 0;
      if constexpr (B == 3 || B == 5 || B == 6) {
        const uint32_t wb = comp(c < 4 ? B0 : B1, c & 3);
        lo = fshr(wa, wb, off);
        hi = wb >> off;
      } else if constexpr (B == 2) {
        lo = wa >> off;
      } else if constexpr (B == 8) {
        hi = comp(c < 4 ? B0 : B1, c & 3);
      }
      unpack8<B>(lo, hi, P[h]);
      const uint32_t s2 = scale_x2(sc, c);
#pragma unroll
      for (int i = 0; i < 4; ++i) P[h][i] = hmul2(P[h][i], s2);  // w = fp16_RN((q - z) s)
    }
    mma_pair<MT>(acc, nt, P[0], P[1], xb0, xb1);
  }
}

// GPTQ half step: exact fp16 (q - z), scaled once: w = fp16_RN((q - z) s);
// zlo / zhi / s2 point at the half's 8 column constants
template <int MT>
__device__ __forceinline__ void gptq_half(const uint4& A0, const uint4& A1, const uint32_t* zlo, const uint32_t* zhi,
                                          const uint32_t* s2, const uint4& xb0, const uint4& xb1,
                                          float (&acc)[MT][4][4]) {
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    uint32_t P[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 2 * nt + h;
      unpack8_gptq(comp(c < 4 ? A0 : A1, c & 3), zlo[c], zhi[c], P[h]);
#pragma unroll
      for (int i = 0; i < 4; ++i) P[h][i] = hmul2(P[h][i], s2[c]);
    }
    mma_pair<MT>(acc, nt, P[0], P[1], xb0, xb1);
  }
}

__device__ __forceinline__ uint4 ld16(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint2 ld8(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint32_t ld4(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// ---------------------------------------------------------------- the kernel

// Fetch side of one warp: walks the CTA's pieces and, inside each, the warp's
// step range, P - 1 steps ahead of the math.
struct Fetch {
  int p;          // position of the next piece in the CTA's share
  int s, ws, we;  // next step to fetch and its range
  int tile;
  bool live;      // a step remains to fetch
};

// Act-order gather: xp[m][j] = x[m][perm[j]] (stored-row order), one element
// per thread so that many loads are in flight. Out-of-range entries read as 0
// and are reported.
__global__ void __launch_bounds__(256) gather_x_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                                                       int M, int K, uint16_t* __restrict__ xp) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  const bool in = e < M * K;
  const int j = in ? e % K : 0;
  const int p = in ? __ldg(perm + j) : 0;  // the permutation is model state: read it before the wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!in) return;
  const bool ok = static_cast<unsigned>(p) < static_cast<unsigned>(K);
  if (!ok) atomicOr(&g_gemv_err, kDevErrBadPerm);
  xp[e] = ok ? __ldg(x + static_cast<size_t>(e / K) * K + p) : static_cast<uint16_t>(0);
}

template <int FMT, int MODE>
__global__ void __launch_bounds__(warps_of(MODE) * 32, 1) gemv_kernel(const __grid_constant__ GemvArgs a) {
  constexpr int NW = warps_of(MODE);
  constexpr int NT = NW * 32;
  constexpr int MT = MODE == 1 ? 2 : 1;
  constexpr int KG = NW / kCG;  // K groups

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* slots = smem;  // [kP][NT][kSlotBytes]
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + a.off_flags);
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + a.off_x);
  uint32_t* meta = reinterpret_cast<uint32_t*>(smem + a.off_meta);
  float* red = reinterpret_cast<float*>(smem + a.off_red);

  const int tid = threadIdx.x;
  const int w = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int cgi = w % kCG, kg = w / kCG;  // the warp's 64-column group and K group

  Split sp;
  sp.total = a.total;
  sp.G = static_cast<int>(gridDim.x);
  sp.n_tiles = a.n_tiles;
  sp.n_steps = a.n_steps;
  sp.kc_steps = a.kc_steps;
  sp.n_chunks = a.n_chunks;
  const int cta = blockIdx.x;
  const int p_begin = sp.begin(cta), p_end = sp.begin(cta + 1);
  const uint32_t nwr = static_cast<uint32_t>(a.n_word_rows);

  // EXL2 step table of the staged chunk: word-row offset | width << 24, or 0
  // for a width outside {2,3,4,5,6,8} or past the end of qweight
  int st_lo = 0, st_hi = 0;
  auto pack_step = [&](uint32_t o, uint32_t e) -> uint32_t {
    o = min(o, nwr);
    e = min(e, nwr);
    const int b = static_cast<int>(e) - static_cast<int>(o);
    const bool ok = b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8;
    return ok ? (o | (static_cast<uint32_t>(b) << 24)) : 0u;
  };
  auto step_of = [&](int s) -> uint32_t {
    if (s >= st_lo && s < st_hi) return meta[s - st_lo];
    return pack_step(__ldg(a.seg_off + s), __ldg(a.seg_off + s + 1));
  };
  auto stage_meta = [&](int kc) {
    st_lo = kc * a.kc_steps;
    st_hi = st_lo + sp.chunk_len(kc);
    if constexpr (FMT == EXQ_FMT_EXL2) {
      for (int i = tid; i < st_hi - st_lo; i += NT)
        meta[i] = pack_step(__ldg(a.seg_off + st_lo + i), __ldg(a.seg_off + st_lo + i + 1));
    }
  };

  // ---- fetch side: one commit group per step, P - 1 steps ahead
  Fetch fs;
  fs.p = p_begin;
  fs.live = false;
  auto fetch_next_range = [&]() {
    fs.live = false;
    while (fs.p < p_end) {
      int next;
      const Piece pc = piece_at(sp, cta, fs.p, p_end, next);
      fs.p = next;
      int ws, we;
      warp_range<KG>(pc, kg, ws, we);
      if (ws < we) {
        fs.s = fs.ws = ws;
        fs.we = we;
        fs.tile = pc.tile;
        fs.live = true;
        return;
      }
    }
  };
  const uint32_t slot0 = smem_u32(slots) + static_cast<uint32_t>(tid * kSlotBytes);
  int iq = 0;  // steps fetched (including empty groups)
  auto fetch = [&]() {
    if (fs.live) {
      const int s = fs.s;
      const int col = fs.tile * kTN + 64 * cgi + 4 * g;
      const bool hi_ok = col + 32 < a.N;  // N % 8 == 0: a 4-column chunk is all in or all out
      const uint32_t dst = slot0 + static_cast<uint32_t>((iq % kP) * NT * kSlotBytes);
      if (col < a.N) {
        if constexpr (FMT == EXQ_FMT_GPTQ4) {
          const uint32_t* src = a.qweight + static_cast<size_t>(4 * s + t) * a.N + col;
          cp_async16(dst, src);
          if (hi_ok) cp_async16(dst + 16, src + 32);
          if (s == fs.ws || s % a.gs_steps == 0) {  // scales and zeros once per group
            const int grp = s / a.gs_steps;
            const uint16_t* sp_ = a.scales + static_cast<size_t>(grp) * a.N + col;
            const uint32_t* zp = a.qzeros + static_cast<size_t>(grp) * (a.N / 8) + col / 8;
            cp_async8(dst + 64, sp_);
            cp_async4(dst + 32, zp);
            if (hi_ok) {
              cp_async8(dst + 72, sp_ + 32);
              cp_async4(dst + 36, zp + 4);
            }
          }
        } else {
          const uint32_t md = step_of(s);
          const int b = static_cast<int>(md >> 24);
          if (b != 0) {
            int wi, off;
            block_window(b, t, wi, off);
            const uint32_t* src = a.qweight + static_cast<size_t>((md & 0xFFFFFFu) + wi) * a.N + col;
            const uint16_t* sp_ = a.scales + static_cast<size_t>(s) * a.N + col;
            const bool second = b == 8 || ((b == 3 || b == 5 || b == 6) && block_needs_second(b, off));
            cp_async16(dst, src);
            if (second) cp_async16(dst + 32, src + a.N);
            cp_async8(dst + 64, sp_);
            if (hi_ok) {
              cp_async16(dst + 16, src + 32);
              if (second) cp_async16(dst + 48, src + a.N + 32);
              cp_async8(dst + 72, sp_ + 32);
            }
          }
        }
      }
      if (++fs.s == fs.we) fetch_next_range();
    }
    cp_async_commit();  // one group per call, possibly empty, keeps the count uniform
    ++iq;
  };

  // ---- staging of x (already in stored-row order), each 8-row block as
  // (x0,x4),(x1,x5),(x2,x6),(x3,x7)
  int next0 = 0;
  const int kc0 = p_begin < p_end ? piece_at(sp, cta, p_begin, p_end, next0).kc : 0;
  auto stage_x = [&](int kc) {
    const int c0 = kc * a.kc_steps;
    const int blocks = sp.chunk_len(kc) * 4;
    const int xtotal = a.M * blocks;
    for (int e = tid; e < xtotal; e += NT) {
      const int m = e / blocks, blk = e - m * blocks;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(m) * a.K + c0 * 32 + blk * 8));
      uint4 o;
      o.x = prmt(v.x, v.z, 0x5410);
      o.y = prmt(v.x, v.z, 0x7632);
      o.z = prmt(v.y, v.w, 0x5410);
      o.w = prmt(v.y, v.w, 0x7632);
      *reinterpret_cast<uint4*>(xs + m * a.xs_stride + blk * 8) = o;
    }
  };

  // weights, scales and offsets are model state: start fetching before the
  // wait for the previous kernel
  if (tid == 0) *last_flag = 0;
  stage_meta(kc0);
  __syncthreads();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  fetch_next_range();
#pragma unroll
  for (int i = 0; i < kP - 1; ++i) fetch();

  asm volatile("griddepcontrol.wait;" ::: "memory");
  int staged = kc0;
  if (p_begin < p_end) stage_x(kc0);
  cta_barrier<NW>();

  int cq = 0;  // steps consumed
  float acc[MT][4][4];
  const uint16_t* xr0 = xs + g * a.xs_stride + 8 * t;
  const uint16_t* xr1 = xs + (g + 8) * a.xs_stride + 8 * t;
  const bool x0_ok = g < a.M, x1_ok = MT == 2 && g + 8 < a.M;
  const uint8_t* myslot = slots + tid * kSlotBytes;

  int p = p_begin, next = p_begin;
  while (p < p_end) {
    const Piece pc = piece_at(sp, cta, p, p_end, next);
    p = next;
    if (pc.kc != staged) {
      cta_barrier<NW>();
      stage_meta(pc.kc);
      stage_x(pc.kc);
      cta_barrier<NW>();
      staged = pc.kc;
    }
    const int c0 = pc.kc * a.kc_steps;
    zero_acc<MT>(acc);
    int ws, we;
    warp_range<KG>(pc, kg, ws, we);

    uint32_t zlo[8], zhi[8], s2[8];  // GPTQ: the current group's column constants
    for (int s = ws; s < we; ++s) {
      fetch();
      cp_async_wait<kP - 1>();  // this lane's copies of step s have landed
      const uint8_t* sl = myslot + (cq % kP) * NT * kSlotBytes;
      ++cq;
      const int kl = (s - c0) * 32;
      const uint4 zero4 = make_uint4(0, 0, 0, 0);
      const uint4 xb0 = x0_ok ? *reinterpret_cast<const uint4*>(xr0 + kl) : zero4;
      const uint4 xb1 = x1_ok ? *reinterpret_cast<const uint4*>(xr1 + kl) : zero4;
      if constexpr (FMT == EXQ_FMT_GPTQ4) {
        if (s == ws || s % a.gs_steps == 0) {  // first step of the warp's part of a group
          const uint32_t zsh = 16u * (g & 1);
          const uint32_t z0 = ld4(sl + 32) >> zsh, z1 = ld4(sl + 36) >> zsh;
#pragma unroll
          for (int c = 0; c < 8; ++c) gptq_zero_consts(((c < 4 ? z0 : z1) >> (4 * (c & 3))) & 0xFu, zlo[c], zhi[c]);
          const uint2 q0 = ld8(sl + 64), q1 = ld8(sl + 72);
          const uint4 sv = make_uint4(q0.x, q0.y, q1.x, q1.y);
#pragma unroll
          for (int c = 0; c < 8; ++c) s2[c] = scale_x2(sv, c);
        }
        gptq_half<MT>(ld16(sl), ld16(sl + 16), zlo, zhi, s2, xb0, xb1, acc);
      } else {
        const uint32_t md = step_of(s);
        const int b = static_cast<int>(md >> 24);
        if (b == 0) {  // warp-uniform; nothing was fetched for it
          if (lane == 0) atomicOr(&g_gemv_err, kDevErrBadSegment);
          continue;
        }
        int wi, off;
        block_window(b, t, wi, off);
        const uint4 A0 = ld16(sl), A1 = ld16(sl + 16);
        const uint4 B0 = ld16(sl + 32), B1 = ld16(sl + 48);
        const uint2 q0 = ld8(sl + 64), q1 = ld8(sl + 72);
        const uint4 sc = make_uint4(q0.x, q0.y, q1.x, q1.y);
        switch (b) {
          case 2: exl2_half<2, MT>(A0, A1, B0, B1, sc, off, xb0, xb1, acc); break;
          case 3: exl2_half<3, MT>(A0, A1, B0, B1, sc, off, xb0, xb1, acc); break;
          case 4: exl2_half<4, MT>(A0, A1, B0, B1, sc, off, xb0, xb1, acc); break;
          case 5: exl2_half<5, MT>(A0, A1, B0, B1, sc, off, xb0, xb1, acc); break;
          case 6: exl2_half<6, MT>(A0, A1, B0, B1, sc, off, xb0, xb1, acc); break;
          default: exl2_half<8, MT>(A0, A1, B0, B1, sc, off, xb0, xb1, acc); break;
        }
      }
    }

    // ---- the piece's sums: K groups added in order, then y or the workspace
    const int elems = a.M * kTN;
    {
      float* rw = red + w * a.M * 64;  // [NW][M][64]
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int m = 8 * mt + 2 * t + (i & 1);
            if (m < a.M) rw[m * 64 + group_col(2 * nt + (i >> 1), g)] = acc[mt][nt][i];
          }
    }
    cta_barrier<NW>();
    // element e = m * kTN + c of the tile: column group c / 64, K groups kg
    auto tile_sum = [&](int e) {
      const int m = e / kTN, c = e - m * kTN;
      float v = 0.f;
      for (int k = 0; k < KG; ++k) v += red[((k * kCG + c / 64) * a.M + m) * 64 + (c & 63)];
      return v;
    };
    const int n0 = pc.tile * kTN;
    if (pc.P == 1) {
      for (int e = tid; e < elems; e += NT) {
        const float v = tile_sum(e);
        const int n = n0 + (e % kTN);
        if (n < a.N) a.y[static_cast<size_t>(e / kTN) * a.N + n] = __half_as_ushort(__float2half_rn(v));
      }
    } else {
      float* part = a.partials + (static_cast<size_t>(pc.tile) * a.max_pieces + pc.slot) * elems;
      for (int e = tid; e < elems; e += NT) part[e] = tile_sum(e);
      __threadfence();
      cta_barrier<NW>();
      if (tid == 0) {
        const unsigned old = atomicAdd(&a.counters[pc.tile], 1u);
        const int last = old == static_cast<unsigned>(pc.P - 1);
        if (last) atomicExch(&a.counters[pc.tile], 0u);  // ready for the next call
        __threadfence();
        *last_flag = last;
      }
      cta_barrier<NW>();
      if (*last_flag) {
        const float* base = a.partials + static_cast<size_t>(pc.tile) * a.max_pieces * elems;
        for (int e = tid; e < elems; e += NT) {
          float v = 0.f;
          for (int k = 0; k < pc.P; ++k) v += __ldcg(base + static_cast<size_t>(k) * elems + e);
          const int n = n0 + (e % kTN);
          if (n < a.N) a.y[static_cast<size_t>(e / kTN) * a.N + n] = __half_as_ushort(__float2half_rn(v));
        }
      }
    }
    cta_barrier<NW>();  // red and last_flag are rewritten by the next piece
  }
  cp_async_wait<0>();
}

}  // namespace
}  // namespace exq

// ================================================================ host side

namespace exq {
namespace {

using KernelFn = void (*)(GemvArgs);

template <int FMT>
KernelFn pick_for(int M) {
  return mode_for(M) == 0 ? gemv_kernel<FMT, 0> : gemv_kernel<FMT, 1>;
}

KernelFn pick_kernel(int fmt, int M) {
  return fmt == EXQ_FMT_GPTQ4 ? pick_for<EXQ_FMT_GPTQ4>(M) : pick_for<EXQ_FMT_EXL2>(M);
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int xs_stride_for(int k_len) {
  // token rows an odd multiple of 64 bytes apart: the quarter-warp of an
  // LDS.128 (two token rows x four 16-byte blocks) touches distinct banks
  return (k_len % 64 == 32) ? k_len : k_len + 32;
}

struct Plan {
  int G, NW, n_tiles, n_steps, kc_steps, n_chunks, max_pieces, xs_stride;
  int total;
  int off_flags, off_x, off_meta, off_red;
  size_t smem;          // dynamic shared memory bytes (with the alignment slack)
  size_t ws_counters;   // bytes of the counter region (256-aligned)
  size_t ws_partials;   // bytes of the partial sums
  size_t ws_bytes;      // workspace bytes (+ M * K * 2 for a permuted layer's gathered x)
};

// Layout of one launch on a device with `sm_count` SMs; false if it cannot fit.
bool make_plan(int K, int N, int M, bool perm, int sm_count, int smem_max, Plan& p) {
  p.n_steps = K / 32;
  p.n_tiles = (N + kTN - 1) / kTN;
  const long long total = static_cast<long long>(p.n_tiles) * p.n_steps;
  if (total >= (1ll << 31)) return false;
  p.total = static_cast<int>(total);
  const int mode = mode_for(M);
  p.NW = warps_of(mode);
  int G = sm_count;
  if (const char* env = std::getenv("EXQ_GEMV_CTAS")) {  // CTA-count override for tuning sweeps
    const int v = std::atoi(env);
    if (v > 0) G = v;
  }
  p.G = std::min(G, p.total);

  size_t off = 0;
  off += static_cast<size_t>(kP) * p.NW * 32 * kSlotBytes;
  p.off_flags = static_cast<int>(off);
  off += 128;
  p.off_red = static_cast<int>(off);
  off += static_cast<size_t>(p.NW) * M * 64 * 4;
  const size_t fixed = off + 1024;  // + slack to align the dynamic base to 1024
  if (fixed >= static_cast<size_t>(smem_max)) return false;
  // x costs M * 64 bytes per step (+ one 64-byte pad per token row), the
  // EXL2 offsets 4 bytes per step (+ 1 entry)
  const long long budget = static_cast<long long>(smem_max) - static_cast<long long>(fixed) - 64LL * M - 64;
  const long long per_step = 64LL * M + 4;
  long long kc = budget / per_step;
  if (kc < 1) return false;
  kc = std::min<long long>(kc, p.n_steps);
  p.n_chunks = static_cast<int>((p.n_steps + kc - 1) / kc);
  p.kc_steps = (p.n_steps + p.n_chunks - 1) / p.n_chunks;  // even chunks
  p.xs_stride = xs_stride_for(p.kc_steps * 32);
  p.off_x = static_cast<int>(off);
  off += align_up(static_cast<size_t>(M) * p.xs_stride * 2, 16);
  p.off_meta = static_cast<int>(off);
  off += align_up(static_cast<size_t>(p.kc_steps + 1) * 4, 16);
  p.smem = off + 1024;
  if (p.smem > static_cast<size_t>(smem_max)) return false;

  // pieces per tile: a unit of len positions meets at most (len - 1) / s + 2
  // shares when every share holds at least s positions
  const int min_share = p.total / p.G;
  p.max_pieces = 0;
  for (int kc_i = 0; kc_i < p.n_chunks; ++kc_i) {
    const int len = kc_i == p.n_chunks - 1 ? p.n_steps - kc_i * p.kc_steps : p.kc_steps;
    p.max_pieces += static_cast<int>((len - 1) / min_share) + 2;
  }
  if (p.n_tiles * 4 > kCounterBytes) return false;
  p.ws_counters = kCounterBytes;  // a fixed region: no call's scratch ever lands on another's counters
  p.ws_partials = align_up(static_cast<size_t>(p.n_tiles) * p.max_pieces * M * kTN * 4, 256);
  p.ws_bytes = p.ws_counters + p.ws_partials + (perm ? align_up(static_cast<size_t>(M) * K * 2, 256) : 0);
  return true;
}

std::mutex g_attr_mutex;
bool g_attr_done[64][4];

}  // namespace

size_t gemv_workspace_bytes(const exq_weight& w, int M) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const DeviceInfo& di = device_info(dev);
  Plan plan{};
  if (!make_plan(w.K, w.N, M, w.perm != nullptr, di.sm_count, di.max_smem_optin, plan)) return 0;
  return plan.ws_bytes;
}

exq_status launch_gemv(const exq_weight& w, const uint16_t* x, int M, uint16_t* y, void* workspace,
                       size_t ws_bytes, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EXQ_ERR_CUDA;
  const DeviceInfo& di = device_info(dev);
  if (di.sm_count <= 0 || dev >= 64) return EXQ_ERR_CUDA;

  Plan plan{};
  if (!make_plan(w.K, w.N, M, w.perm != nullptr, di.sm_count, di.max_smem_optin, plan)) return EXQ_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < plan.ws_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return EXQ_ERR_INVALID_ARG;

  KernelFn fn = pick_kernel(w.format, M);
  const int fidx = (w.format == EXQ_FMT_GPTQ4 ? 0 : 2) + mode_for(M);
  {
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    if (!g_attr_done[dev][fidx]) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin) != cudaSuccess)
        return EXQ_ERR_CUDA;
      g_attr_done[dev][fidx] = true;
    }
  }

  static const bool no_pdl = std::getenv("EXQ_NO_PDL") != nullptr;
  cudaLaunchAttribute attrs[1];
  int na = 0;
  if (!no_pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }

  // act-order: gather x into stored-row order once, into the workspace
  const uint16_t* xs_src = x;
  if (w.perm) {
    uint16_t* xp = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + plan.ws_counters +
                                               plan.ws_partials);
    const int threads = M * w.K;
    cudaLaunchConfig_t gcfg{};
    gcfg.gridDim = dim3((threads + 255) / 256, 1, 1);
    gcfg.blockDim = dim3(256, 1, 1);
    gcfg.stream = stream;
    gcfg.attrs = attrs;
    gcfg.numAttrs = na;
    if (cudaLaunchKernelEx(&gcfg, gather_x_kernel, x, w.perm, M, w.K, xp) != cudaSuccess) {
      cudaGetLastError();
      return EXQ_ERR_CUDA;
    }
    xs_src = xp;
  }

  GemvArgs args{};
  args.qweight = w.qweight;
  args.scales = w.scales;
  args.qzeros = w.qzeros;
  args.seg_off = w.seg_word_off;
  args.x = xs_src;
  args.y = y;
  args.counters = static_cast<uint32_t*>(workspace);
  args.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan.ws_counters);
  args.K = w.K;
  args.N = w.N;
  args.M = M;
  args.n_steps = plan.n_steps;
  args.gs_steps = w.format == EXQ_FMT_GPTQ4 ? w.group_size / 32 : 1;
  args.n_word_rows = w.n_word_rows;
  args.n_tiles = plan.n_tiles;
  args.kc_steps = plan.kc_steps;
  args.n_chunks = plan.n_chunks;
  args.max_pieces = plan.max_pieces;
  args.xs_stride = plan.xs_stride;
  args.total = plan.total;
  args.off_flags = plan.off_flags;
  args.off_x = plan.off_x;
  args.off_meta = plan.off_meta;
  args.off_red = plan.off_red;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(plan.G, 1, 1);
  cfg.blockDim = dim3(plan.NW * 32, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, fn, args) != cudaSuccess) {
    cudaGetLastError();
    return EXQ_ERR_CUDA;
  }
  return EXQ_OK;
}

unsigned take_gemv_errors(cudaStream_t stream) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_gemv_err, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return ~0u;
  if (cudaMemcpyToSymbolAsync(g_gemv_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return ~0u;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ~0u;
  return v;
}

}  // namespace exq
