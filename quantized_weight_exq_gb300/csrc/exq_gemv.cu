// Decode-sized fused quantized matmul, 1 <= M <= 16:  y = x . dequant(Wq).
//
// Follows the fused kernel of the ExLlamaV2 blog post ("ExLlamaV2: The fastest
// inference engine for quantized Llama/HF models", section "How the Fused CUDA
// Kernel Works"): packed weights are streamed from memory once, unpacked and
// scaled in registers, multiplied into fp32 sums and written as fp16. The
// act-order row remapping (ExLlamaV2 README, "EXL2 quantization") is applied
// to x while it is staged in shared memory, so the weights stream in stored
// order.
//
// GB300 mapping:
//  * Persistent CTAs (one per SM, 16 warps). A thread-block cluster of C CTAs
//    splits K; each cluster walks column tiles of TN = 64 * CG columns, and
//    the CTA's 16 warps form CG column groups x (16 / CG) K groups. x for the
//    CTA's K range is gathered (through the permutation) into shared memory
//    once and reused for every tile.
//  * Per 32-row step a lane (g = lane / 4, t = lane % 4) owns 8 adjacent
//    columns of the rows [8t, 8t + 8): two 128-bit loads per word row, so 8
//    lanes read 256 contiguous bytes. Register slots keep several steps of
//    loads in flight, and the pipeline runs on across tile boundaries.
//  * Dequantised fp16 pairs feed mma.sync m16n8k16 (fp16 in, fp32 accumulate)
//    with swapped roles: A = W^T (16 columns x 16 K), B = x^T (16 K x 8
//    tokens). The K order inside a 16-slab is free as long as A and B agree,
//    so x is staged in the pair order the unpackers produce.
//  * Reduction per tile: warps of a K group through shared memory, then the
//    CTAs of the cluster through distributed shared memory in rank order --
//    deterministic, no workspace.
//  * Programmatic dependent launch: the kernel lets the next launch start
//    early and issues its first weight loads before waiting for the previous
//    kernel; x is read and y written only after that wait.
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

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;

struct GemvArgs {
  const uint32_t* qweight;
  const uint16_t* scales;
  const uint32_t* qzeros;
  const int32_t* perm;
  const uint32_t* seg_off;
  const uint16_t* x;
  uint16_t* y;
  int K, N, M;
  int n_steps;      // K / 32
  int gs_steps;     // GPTQ: group_size / 32
  int gs_shift;     // log2(gs_steps) when it is a power of two, else -1
  int n_word_rows;  // rows of qweight (bound for EXL2 segment tables)
  int cg;           // 64-column groups per CTA tile (1, 2 or 4)
  int cta_steps;    // steps per cluster rank
  int warp_steps;   // steps per K-group warp, a multiple of the prefetch depth
  int n_tiles;      // ceil(N / (64 * cg))
  int xs_stride;    // halves per staged x row
};

__device__ __forceinline__ uint4 ld_stream(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// column c (0..7) of a pair of 4-column vectors
__device__ __forceinline__ uint32_t col8(const uint4 (&v)[2], int c) { return comp(v[c >> 2], c & 3); }

// fp16 scale of column c as (s, s)
__device__ __forceinline__ uint32_t scale2(const uint4& sc, int c) {
  const uint32_t h = comp(sc, c >> 1);
  return (c & 1) ? prmt(h, h, 0x3232) : prmt(h, h, 0x1010);
}

// one step's loads for one lane
template <int FMT>
struct Slot;

template <>
struct Slot<EXQ_FMT_GPTQ4> {
  uint4 w[2];     // word row 4s + t, 8 columns
  uint4 sc;       // 8 fp16 scales of the step's group
  uint32_t zw;    // 8 zero nibbles
  int fresh;      // first step of a group (or of the warp's range): rebuild constants
};

template <>
struct Slot<EXQ_FMT_EXL2> {
  uint4 wa[2], wb[2];  // first / second word row of the lane's block
  uint4 sc;            // 8 fp16 scales of the step's segment
  int bits, off;       // width of the segment (0 = skip), bit offset of the block
};

__device__ __forceinline__ void zero_slot(Slot<EXQ_FMT_GPTQ4>& sl) {
  sl.w[0] = sl.w[1] = make_uint4(0, 0, 0, 0);
  sl.sc = make_uint4(0, 0, 0, 0);
  sl.zw = 0;
  sl.fresh = 1;
}

__device__ __forceinline__ void zero_slot(Slot<EXQ_FMT_EXL2>& sl) {
  sl.wa[0] = sl.wa[1] = sl.wb[0] = sl.wb[1] = make_uint4(0, 0, 0, 0);
  sl.sc = make_uint4(0, 0, 0, 0);
  sl.bits = 0;
  sl.off = 0;
}

// Step s (absolute) for the lane's columns [col, col + 8). `step_ok` is
// uniform across the warp and decides whether the step is computed at all;
// `col_ok` is per lane and only zeroes the lane's data, so that every lane of
// a warp always reaches the same mma.sync instructions.
__device__ __forceinline__ void load_slot(const GemvArgs& a, const uint32_t*, Slot<EXQ_FMT_GPTQ4>& sl, int s,
                                          int t, int col, bool step_ok, bool col_ok, int cs0, int ws0) {
  (void)cs0;
  if (!step_ok) {
    zero_slot(sl);
    return;
  }
  const int grp = a.gs_shift >= 0 ? (s >> a.gs_shift) : s / a.gs_steps;
  sl.fresh = (s == ws0) || (s - grp * a.gs_steps == 0);
  if (!col_ok) {
    sl.w[0] = sl.w[1] = make_uint4(0, 0, 0, 0);
    sl.sc = make_uint4(0, 0, 0, 0);
    sl.zw = 0;
    return;
  }
  const uint32_t* p = a.qweight + static_cast<size_t>(4 * s + t) * a.N + col;
  sl.w[0] = ld_stream(p);
  sl.w[1] = ld_stream(p + 4);
  sl.sc = __ldg(reinterpret_cast<const uint4*>(a.scales + static_cast<size_t>(grp) * a.N + col));
  sl.zw = __ldg(a.qzeros + static_cast<size_t>(grp) * (a.N >> 3) + (col >> 3));
}

__device__ __forceinline__ void load_slot(const GemvArgs& a, const uint32_t* meta, Slot<EXQ_FMT_EXL2>& sl, int s,
                                          int t, int col, bool step_ok, bool col_ok, int cs0, int) {
  const uint32_t md = step_ok ? meta[s - cs0] : 0u;  // same for every lane of the warp
  const int b = static_cast<int>(md >> 24);
  if (b == 0 || !col_ok) {
    zero_slot(sl);
    sl.bits = b;
    return;
  }
  int wi, off;
  block_window(b, t, wi, off);
  const uint32_t* p = a.qweight + static_cast<size_t>((md & 0xFFFFFFu) + wi) * a.N + col;
  sl.wa[0] = ld_stream(p);
  sl.wa[1] = ld_stream(p + 4);
  if (block_needs_second(b, off)) {
    sl.wb[0] = ld_stream(p + a.N);
    sl.wb[1] = ld_stream(p + a.N + 4);
  } else {
    sl.wb[0] = sl.wb[1] = make_uint4(0, 0, 0, 0);
  }
  sl.sc = __ldg(reinterpret_cast<const uint4*>(a.scales + static_cast<size_t>(s) * a.N + col));
  sl.bits = b;
  sl.off = off;
}

template <int MT>
__device__ __forceinline__ void mma_pair(float (&acc)[MT][4][4], int nt, const uint32_t (&P0)[4],
                                         const uint32_t (&P1)[4], const uint4& xb0, const uint4& xb1) {
  // slab 0: pairs 0 (k 2t, 2t+1) and 1 (k 2t+8, 2t+9); slab 1: pairs 2 and 3
  mma16816(acc[0][nt], P0[0], P1[0], P0[1], P1[1], xb0.x, xb0.y);
  mma16816(acc[0][nt], P0[2], P1[2], P0[3], P1[3], xb0.z, xb0.w);
  if constexpr (MT == 2) {
    mma16816(acc[1][nt], P0[0], P1[0], P0[1], P1[1], xb1.x, xb1.y);
    mma16816(acc[1][nt], P0[2], P1[2], P0[3], P1[3], xb1.z, xb1.w);
  }
}

template <int B, int MT>
__device__ __forceinline__ void exl2_step(const Slot<EXQ_FMT_EXL2>& sl, float (&acc)[MT][4][4], const uint4& xb0,
                                          const uint4& xb1) {
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    uint32_t P[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 2 * nt + h;
      const uint32_t wa = col8(sl.wa, c);
      uint32_t lo = wa, hi = 0;
      if constexpr (B == 3 || B == 5 || B == 6) {  // blocks can start mid-word and spill over
        const uint32_t wb = col8(sl.wb, c);
        lo = fshr(wa, wb, sl.off);
        hi = wb >> sl.off;
      } else if constexpr (B == 2) {  // 16-bit blocks at offset 0 or 16 of one word
        lo = wa >> sl.off;
      } else if constexpr (B == 8) {  // two whole words
        hi = col8(sl.wb, c);
      }
      unpack8<B>(lo, hi, P[h]);
      const uint32_t s2 = scale2(sl.sc, c);
#pragma unroll
      for (int i = 0; i < 4; ++i) P[h][i] = hmul2(P[h][i], s2);
    }
    mma_pair<MT>(acc, nt, P[0], P[1], xb0, xb1);
  }
}

template <int FMT, int MT, bool PERM, int KP>
__global__ void __launch_bounds__(kThreads, 1) gemv_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];

  const int crank = blockIdx.x;  // the cluster spans grid.x
  const int ncta = gridDim.x;
  const int cluster_id = blockIdx.y, n_clusters = gridDim.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int cgi = warp % a.cg, kg = warp / a.cg;
  const int TN = 64 * a.cg;

  const int cs0 = crank * a.cta_steps;
  const int cs1 = min(a.n_steps, cs0 + a.cta_steps);
  const int csn = max(0, cs1 - cs0);
  const int ws0 = cs0 + kg * a.warp_steps;           // warp range [ws0, ws0 + warp_steps) clipped to cs1
  const int ws_end = min(cs1, ws0 + a.warp_steps);

  // shared memory: [x rows][EXL2 segment table][per-warp partials][CTA partials]
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  uint32_t* meta = reinterpret_cast<uint32_t*>(smem + static_cast<size_t>(a.M) * a.xs_stride * 2);
  float* red = reinterpret_cast<float*>(meta + ((a.cta_steps + 3) & ~3));
  float* red2 = red + kWarps * a.M * 64;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if constexpr (FMT == EXQ_FMT_EXL2) {
    // segment table of the CTA range: word-row offset | width << 24 (0 = invalid)
    for (int i = threadIdx.x; i < csn; i += kThreads) {
      const unsigned o0 = __ldg(a.seg_off + cs0 + i), o1 = __ldg(a.seg_off + cs0 + i + 1);
      const int b = static_cast<int>(o1 - o0);
      const bool ok = (b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8) && o1 > o0 &&
                      o1 <= static_cast<unsigned>(a.n_word_rows);
      if (!ok) atomicOr(&g_gemv_err, kDevErrBadSegment);
      meta[i] = ok ? (o0 | (static_cast<uint32_t>(b) << 24)) : 0u;
    }
    __syncthreads();
  }

  // first tile's loads are issued before waiting for the previous kernel
  Slot<FMT> slot[KP];
  {
    const int col = cluster_id * TN + cgi * 64 + 8 * g;
    const bool col_ok = cluster_id < a.n_tiles && col < a.N;
#pragma unroll
    for (int u = 0; u < KP; ++u)
      load_slot(a, meta, slot[u], ws0 + u, t, col, cluster_id < a.n_tiles && ws0 + u < ws_end, col_ok, cs0, ws0);
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");

  // stage x[:, CTA range]: stored-row order, each 8-row block as
  // (x0,x4),(x1,x5),(x2,x6),(x3,x7); all permutation loads first, then x
  {
    const int blocks = csn * 4;
    const int total = a.M * blocks;
    for (int base = 0; base < total; base += 2 * kThreads) {
      uint32_t w[2][4];
      int dst[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int e = base + r * kThreads + threadIdx.x;
        dst[r] = -1;
        if (e < total) {
          const int m = e / blocks, blk = e - m * blocks;
          const int k = cs0 * 32 + blk * 8;
          const uint16_t* xr = a.x + static_cast<size_t>(m) * a.K;
          dst[r] = m * a.xs_stride + blk * 8;
          if constexpr (PERM) {
            const int4 p0 = __ldg(reinterpret_cast<const int4*>(a.perm + k));
            const int4 p1 = __ldg(reinterpret_cast<const int4*>(a.perm + k + 4));
            w[r][0] = __ldg(xr + p0.x) | (static_cast<uint32_t>(__ldg(xr + p0.y)) << 16);
            w[r][1] = __ldg(xr + p0.z) | (static_cast<uint32_t>(__ldg(xr + p0.w)) << 16);
            w[r][2] = __ldg(xr + p1.x) | (static_cast<uint32_t>(__ldg(xr + p1.y)) << 16);
            w[r][3] = __ldg(xr + p1.z) | (static_cast<uint32_t>(__ldg(xr + p1.w)) << 16);
          } else {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + k));
            w[r][0] = v.x; w[r][1] = v.y; w[r][2] = v.z; w[r][3] = v.w;
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        if (dst[r] >= 0) {
          uint4 o;
          o.x = prmt(w[r][0], w[r][2], 0x5410);
          o.y = prmt(w[r][0], w[r][2], 0x7632);
          o.z = prmt(w[r][1], w[r][3], 0x5410);
          o.w = prmt(w[r][1], w[r][3], 0x7632);
          *reinterpret_cast<uint4*>(xs + dst[r]) = o;
        }
      }
    }
  }
  __syncthreads();

  float acc[MT][4][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;

  uint32_t s2[8], zlo[8], zhi[8];
  const uint32_t red_s = static_cast<uint32_t>(__cvta_generic_to_shared(red2));

  for (int tile = cluster_id; tile < a.n_tiles; tile += n_clusters) {
    for (int jb = 0; jb < a.warp_steps; jb += KP) {
#pragma unroll
      for (int u = 0; u < KP; ++u) {
        const int j = jb + u;
        const int s = ws0 + j;
        Slot<FMT>& sl = slot[u];
        if (s < ws_end) {  // warp-uniform: every lane runs the same mma.sync sequence
          const int kl = (s - cs0) * 32 + 8 * t;
          uint4 xb0 = make_uint4(0, 0, 0, 0), xb1 = make_uint4(0, 0, 0, 0);
          if (g < a.M) xb0 = *reinterpret_cast<const uint4*>(xs + g * a.xs_stride + kl);
          if (MT == 2 && g + 8 < a.M) xb1 = *reinterpret_cast<const uint4*>(xs + (g + 8) * a.xs_stride + kl);
          if constexpr (FMT == EXQ_FMT_GPTQ4) {
            if (sl.fresh) {
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                gptq_zero_consts((sl.zw >> (4 * c)) & 0xFu, zlo[c], zhi[c]);
                s2[c] = scale2(sl.sc, c);
              }
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
              uint32_t P[2][4];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int c = 2 * nt + h;
                unpack8_gptq(col8(sl.w, c), zlo[c], zhi[c], P[h]);
#pragma unroll
                for (int i = 0; i < 4; ++i) P[h][i] = hmul2(P[h][i], s2[c]);
              }
              mma_pair<MT>(acc, nt, P[0], P[1], xb0, xb1);
            }
          } else {
            switch (sl.bits) {
              case 2: exl2_step<2, MT>(sl, acc, xb0, xb1); break;
              case 3: exl2_step<3, MT>(sl, acc, xb0, xb1); break;
              case 4: exl2_step<4, MT>(sl, acc, xb0, xb1); break;
              case 5: exl2_step<5, MT>(sl, acc, xb0, xb1); break;
              case 6: exl2_step<6, MT>(sl, acc, xb0, xb1); break;
              case 8: exl2_step<8, MT>(sl, acc, xb0, xb1); break;
              default: break;  // invalid segment: contributes nothing (reported above)
            }
          }
        }
        // refill: step j + KP of this tile, or the first steps of the next one
        int nj = j + KP, ntile = tile;
        if (nj >= a.warp_steps) {
          nj -= a.warp_steps;
          ntile += n_clusters;
        }
        const int ncol = ntile * TN + cgi * 64 + 8 * g;
        load_slot(a, meta, sl, ws0 + nj, t, ncol, ntile < a.n_tiles && ws0 + nj < ws_end, ncol < a.N, cs0, ws0);
      }
    }

    // ---- tile reduction: K-group warps (smem), then cluster ranks (DSMEM)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const int m0 = 8 * mt + 2 * t, c0 = 8 * g + 2 * nt;
        float* r = red + warp * a.M * 64;
        if (m0 < a.M) {
          r[m0 * 64 + c0] = acc[mt][nt][0];
          r[m0 * 64 + c0 + 1] = acc[mt][nt][2];
        }
        if (m0 + 1 < a.M) {
          r[(m0 + 1) * 64 + c0] = acc[mt][nt][1];
          r[(m0 + 1) * 64 + c0 + 1] = acc[mt][nt][3];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;
      }
    __syncthreads();
    const int kgroups = kWarps / a.cg;
    const int elems = a.M * TN;
    if (ncta == 1) {
      for (int e = threadIdx.x; e < elems; e += kThreads) {
        const int m = e / TN, c = e - m * TN;
        const int cg = c >> 6, cc = c & 63;
        float v = 0.f;
        for (int k = 0; k < kgroups; ++k) v += red[((k * a.cg + cg) * a.M + m) * 64 + cc];
        const int n = tile * TN + c;
        if (n < a.N) a.y[static_cast<size_t>(m) * a.N + n] = __half_as_ushort(__float2half_rn(v));
      }
    } else {
      for (int e = threadIdx.x; e < elems; e += kThreads) {
        const int m = e / TN, c = e - m * TN;
        const int cg = c >> 6, cc = c & 63;
        float v = 0.f;
        for (int k = 0; k < kgroups; ++k) v += red[((k * a.cg + cg) * a.M + m) * 64 + cc];
        red2[e] = v;
      }
      asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
      for (int e = crank + ncta * threadIdx.x; e < elems; e += ncta * kThreads) {
        float v = 0.f;
        for (int r = 0; r < ncta; ++r) {
          uint32_t remote;
          float pv;
          asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(red_s + 4u * e), "r"(r));
          asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(pv) : "r"(remote) : "memory");
          v += pv;
        }
        const int m = e / TN, c = e - m * TN;
        const int n = tile * TN + c;
        if (n < a.N) a.y[static_cast<size_t>(m) * a.N + n] = __half_as_ushort(__float2half_rn(v));
      }
      // red2 of every rank stays alive until all ranks have read it
      asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    }
    __syncthreads();  // red is rewritten by the next tile
  }
}

using KernelFn = void (*)(GemvArgs);

template <int FMT, int MT, bool PERM>
constexpr int kPrefetch = FMT == EXQ_FMT_GPTQ4 ? (MT == 1 ? 4 : 3) : (MT == 1 ? 3 : 2);

template <int FMT, int MT, bool PERM>
KernelFn kernel_ptr() {
  return gemv_kernel<FMT, MT, PERM, kPrefetch<FMT, MT, PERM>>;
}

KernelFn pick_kernel(int fmt, int mt, bool perm, int& kp) {
  if (fmt == EXQ_FMT_GPTQ4) {
    kp = mt == 1 ? 4 : 3;
    if (mt == 1) return perm ? kernel_ptr<EXQ_FMT_GPTQ4, 1, true>() : kernel_ptr<EXQ_FMT_GPTQ4, 1, false>();
    return perm ? kernel_ptr<EXQ_FMT_GPTQ4, 2, true>() : kernel_ptr<EXQ_FMT_GPTQ4, 2, false>();
  }
  kp = mt == 1 ? 3 : 2;
  if (mt == 1) return perm ? kernel_ptr<EXQ_FMT_EXL2, 1, true>() : kernel_ptr<EXQ_FMT_EXL2, 1, false>();
  return perm ? kernel_ptr<EXQ_FMT_EXL2, 2, true>() : kernel_ptr<EXQ_FMT_EXL2, 2, false>();
}

int xs_stride_for(int k_len) {
  // token rows an odd multiple of 64 bytes apart: the quarter-warp of an
  // LDS.128 (two token rows x four 16-byte blocks) touches distinct banks
  return (k_len % 64 == 32) ? k_len : k_len + 32;
}

struct Plan {
  int cg, c, clusters, cta_steps, warp_steps, n_tiles, xs_stride;
  size_t smem;
};

size_t smem_bytes(int M, int cta_steps, int cg, int xs_stride) {
  return static_cast<size_t>(M) * xs_stride * 2 + static_cast<size_t>((cta_steps + 3) & ~3) * 4 +
         static_cast<size_t>(kWarps) * M * 64 * 4 + static_cast<size_t>(M) * 64 * cg * 4;
}

// Choose the tile width (64 * cg columns) and cluster size c (CTAs splitting
// K): one CTA per SM, so clusters = SMs / c; model the time as
// tiles-per-cluster x (steps per warp + a per-tile reduction cost) and keep
// the split that minimises it.
bool make_plan(int K, int N, int M, int kp, int sm_count, int smem_max, Plan& best) {
  const int n_steps = K / 32;
  double best_cost = 1e300;
  bool found = false;
  for (int cg : {4, 2, 1}) {
    const int kgroups = kWarps / cg;
    const int n_tiles = (N + 64 * cg - 1) / (64 * cg);
    for (int c = 1; c <= 8; ++c) {
      const int cta_steps = (n_steps + c - 1) / c;
      if (c > 1 && (c - 1) * cta_steps >= n_steps) break;  // an empty rank
      int warp_steps = (cta_steps + kgroups - 1) / kgroups;
      warp_steps = (warp_steps + kp - 1) / kp * kp;
      const int xs_stride = xs_stride_for(cta_steps * 32);
      const size_t smem = smem_bytes(M, cta_steps, cg, xs_stride);
      if (smem > static_cast<size_t>(smem_max)) continue;
      const int clusters = std::max(1, std::min(n_tiles, sm_count / c));
      const int iters = (n_tiles + clusters - 1) / clusters;
      // a step moves 32 rows x 64 columns per warp; the reduction and its
      // barriers cost roughly a few steps per tile, more with a cluster
      const double cost = iters * (warp_steps + 3.0 + 1.5 * (c > 1) + 0.02 * M * cg) + 0.05 * c;
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = Plan{cg, c, clusters, cta_steps, warp_steps, n_tiles, xs_stride, smem};
        found = true;
      }
    }
  }
  return found;
}

std::mutex g_attr_mutex;
bool g_attr_done[64][8];

}  // namespace

exq_status launch_gemv(const exq_weight& w, const uint16_t* x, int M, uint16_t* y, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EXQ_ERR_CUDA;
  const DeviceInfo& di = device_info(dev);
  if (di.sm_count <= 0 || dev >= 64) return EXQ_ERR_CUDA;
  if (w.n_word_rows >= (1 << 24)) return EXQ_ERR_UNSUPPORTED;

  const int mt = M <= 8 ? 1 : 2;
  const bool perm = w.perm != nullptr;
  int kp = 0;
  KernelFn fn = pick_kernel(w.format, mt, perm, kp);
  const int fidx = (w.format == EXQ_FMT_GPTQ4 ? 0 : 4) + (mt - 1) * 2 + (perm ? 1 : 0);
  {
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    if (!g_attr_done[dev][fidx]) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin) != cudaSuccess)
        return EXQ_ERR_CUDA;
      g_attr_done[dev][fidx] = true;
    }
  }

  Plan plan{};
  if (!make_plan(w.K, w.N, M, kp, di.sm_count, di.max_smem_optin, plan)) return EXQ_ERR_UNSUPPORTED;
  if (const char* env = std::getenv("EXQ_GEMV_PLAN")) {  // "cg,c" override for tuning sweeps
    int cg = 0, c = 0;
    if (std::sscanf(env, "%d,%d", &cg, &c) == 2 && (cg == 1 || cg == 2 || cg == 4) && c >= 1 && c <= 8) {
      const int n_steps = w.K / 32, kgroups = kWarps / cg;
      Plan p{};
      p.cg = cg;
      p.c = c;
      p.n_tiles = (w.N + 64 * cg - 1) / (64 * cg);
      p.clusters = std::max(1, std::min(p.n_tiles, di.sm_count / c));
      p.cta_steps = (n_steps + c - 1) / c;
      p.warp_steps = ((p.cta_steps + kgroups - 1) / kgroups + kp - 1) / kp * kp;
      p.xs_stride = xs_stride_for(p.cta_steps * 32);
      p.smem = smem_bytes(M, p.cta_steps, cg, p.xs_stride);
      if (p.smem <= static_cast<size_t>(di.max_smem_optin) && (c == 1 || (c - 1) * p.cta_steps < n_steps))
        plan = p;
    }
  }

  GemvArgs args{};
  args.qweight = w.qweight;
  args.scales = w.scales;
  args.qzeros = w.qzeros;
  args.perm = w.perm;
  args.seg_off = w.seg_word_off;
  args.x = x;
  args.y = y;
  args.K = w.K;
  args.N = w.N;
  args.M = M;
  args.n_steps = w.K / 32;
  args.gs_steps = w.format == EXQ_FMT_GPTQ4 ? w.group_size / 32 : 1;
  args.gs_shift = (args.gs_steps & (args.gs_steps - 1)) == 0 ? __builtin_ctz(args.gs_steps) : -1;
  args.n_word_rows = w.n_word_rows;
  args.cg = plan.cg;
  args.cta_steps = plan.cta_steps;
  args.warp_steps = plan.warp_steps;
  args.n_tiles = plan.n_tiles;
  args.xs_stride = plan.xs_stride;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(plan.c, plan.clusters, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeClusterDimension;
  attrs[na].val.clusterDim.x = plan.c;
  attrs[na].val.clusterDim.y = 1;
  attrs[na].val.clusterDim.z = 1;
  ++na;
  static const bool no_pdl = std::getenv("EXQ_NO_PDL") != nullptr;
  if (!no_pdl) {
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
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
