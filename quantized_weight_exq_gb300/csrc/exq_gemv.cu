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
//  * A warp owns a 32-column strip and walks 32 stored rows per step
//    (4 word rows of GPTQ, one EXL2 segment). Lane (g = lane/4, t = lane%4)
//    loads one 128-bit vector = 4 adjacent columns of the word row(s) holding
//    rows [8t, 8t+8) of the step, so 8 lanes cover 128 contiguous bytes.
//  * The dequantised fp16 pairs are used directly as the A operand of
//    mma.sync m16n8k16 (fp16 in, fp32 accumulate) with the roles swapped:
//    A = W^T (16 columns x 16 rows of K), B = x^T (16 rows of K x 8 tokens).
//    The order of K inside a 16-slab is free as long as A and B agree, so x
//    is staged in smem in the pair order the unpackers produce.
//  * Split-K: the warps of a CTA split the CTA's K range; the CTAs of a
//    thread-block cluster (<= 8, one strip) split K further and reduce their
//    fp32 partials through distributed shared memory in rank order, so the
//    result is deterministic and no workspace is needed.
//  * Programmatic dependent launch: the kernel lets the next launch start
//    early and prefetches its first weight vectors before waiting for the
//    previous kernel; x is read and y written only after that wait.
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "exq_device.cuh"
#include "exq_internal.h"

namespace exq {
namespace {

__device__ unsigned g_gemv_err;

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kPrefetch = 4;  // steps of weight vectors in flight per lane

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
  int n_word_rows;  // rows of qweight (bounds for EXL2 segment tables)
  int cta_steps;    // steps per CTA (the last one may get fewer)
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

// one step's loads for one lane
struct Slot {
  uint4 wa, wb;    // word row(s) for the lane's 4 columns
  uint2 sc;        // 4 fp16 scales
  uint32_t zw;     // GPTQ: zero word
  int bits, off;   // EXL2: width of the step's segment, bit offset of the lane's block
};

template <int FMT>
__device__ __forceinline__ void load_slot(const GemvArgs& a, Slot& sl, int s, int t, int col, bool col_ok) {
  if constexpr (FMT == EXQ_FMT_GPTQ4) {
    const int grp = s / a.gs_steps;
    sl.wa = col_ok ? ld_stream(a.qweight + static_cast<size_t>(4 * s + t) * a.N + col) : make_uint4(0, 0, 0, 0);
    sl.sc = col_ok ? __ldg(reinterpret_cast<const uint2*>(a.scales + static_cast<size_t>(grp) * a.N + col))
                   : make_uint2(0, 0);
    sl.zw = col_ok ? __ldg(a.qzeros + static_cast<size_t>(grp) * (a.N >> 3) + (col >> 3)) : 0u;
  } else {
    const unsigned o0 = __ldg(a.seg_off + s), o1 = __ldg(a.seg_off + s + 1);
    int b = static_cast<int>(o1 - o0);
    const bool ok = (b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8) && o1 > o0 &&
                    o1 <= static_cast<unsigned>(a.n_word_rows);
    if (!ok) b = 0;
    int wi = 0, off = 0;
    if (ok) block_window(b, t, wi, off);
    const size_t row = static_cast<size_t>(o0) + wi;
    sl.wa = (ok && col_ok) ? ld_stream(a.qweight + row * a.N + col) : make_uint4(0, 0, 0, 0);
    sl.wb = (ok && col_ok && block_needs_second(b, off)) ? ld_stream(a.qweight + (row + 1) * a.N + col)
                                                          : make_uint4(0, 0, 0, 0);
    sl.sc = col_ok ? __ldg(reinterpret_cast<const uint2*>(a.scales + static_cast<size_t>(s) * a.N + col))
                   : make_uint2(0, 0);
    sl.bits = b;
    sl.off = off;
  }
}

template <int B>
__device__ __forceinline__ void exl2_cols(const Slot& sl, const uint32_t (&s2)[4], uint32_t (&P)[4][4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t wa = comp(sl.wa, c), wb = comp(sl.wb, c);
    const uint32_t lo = fshr(wa, wb, sl.off), hi = wb >> sl.off;
    unpack8<B>(lo, hi, P[c]);
#pragma unroll
    for (int i = 0; i < 4; ++i) P[c][i] = hmul2(P[c][i], s2[c]);
  }
}

template <int FMT, int MT, bool PERM>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const __grid_constant__ GemvArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);

  const int crank = blockIdx.x;  // cluster spans grid.x, so this is the rank
  const int ncta = gridDim.x;
  const int strip = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int col = strip * 32 + 4 * g;
  const bool col_ok = col < a.N;

  const int cs0 = crank * a.cta_steps;
  const int cs1 = min(a.n_steps, cs0 + a.cta_steps);
  const int csn = max(0, cs1 - cs0);
  const int ws0 = cs0 + (csn * warp) / kWarps;
  const int ws1 = cs0 + (csn * (warp + 1)) / kWarps;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // weights are model state: start streaming them before the previous
  // kernel on the stream has finished
  Slot slot[kPrefetch];
#pragma unroll
  for (int u = 0; u < kPrefetch; ++u)
    if (ws0 + u < ws1) load_slot<FMT>(a, slot[u], ws0 + u, t, col, col_ok);

  asm volatile("griddepcontrol.wait;" ::: "memory");

  // stage x[:, CTA range] into smem, rows in stored order, each 8-row block
  // as (x0,x4),(x1,x5),(x2,x6),(x3,x7)
  {
    const int blocks = csn * 4;  // 8-row blocks per token row
    const int k0 = cs0 * 32;
    for (int e = threadIdx.x; e < a.M * blocks; e += kThreads) {
      const int m = e / blocks, blk = e - m * blocks;
      const int k = k0 + blk * 8;
      uint32_t w0, w1, w2, w3;
      const uint16_t* xr = a.x + static_cast<size_t>(m) * a.K;
      if constexpr (PERM) {
        const int4 p0 = __ldg(reinterpret_cast<const int4*>(a.perm + k));
        const int4 p1 = __ldg(reinterpret_cast<const int4*>(a.perm + k + 4));
        w0 = __ldg(xr + p0.x) | (static_cast<uint32_t>(__ldg(xr + p0.y)) << 16);
        w1 = __ldg(xr + p0.z) | (static_cast<uint32_t>(__ldg(xr + p0.w)) << 16);
        w2 = __ldg(xr + p1.x) | (static_cast<uint32_t>(__ldg(xr + p1.y)) << 16);
        w3 = __ldg(xr + p1.z) | (static_cast<uint32_t>(__ldg(xr + p1.w)) << 16);
      } else {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + k));
        w0 = v.x; w1 = v.y; w2 = v.z; w3 = v.w;
      }
      uint4 o;
      o.x = prmt(w0, w2, 0x5410);
      o.y = prmt(w0, w2, 0x7632);
      o.z = prmt(w1, w3, 0x5410);
      o.w = prmt(w1, w3, 0x7632);
      *reinterpret_cast<uint4*>(xs + m * a.xs_stride + blk * 8) = o;
    }
  }
  __syncthreads();

  float acc[MT][2][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;

  uint32_t s2[4] = {0, 0, 0, 0}, zlo[4] = {0, 0, 0, 0}, zhi[4] = {0, 0, 0, 0};
  int cur_grp = -1;
  unsigned bad = 0;

  for (int sb = ws0; sb < ws1; sb += kPrefetch) {
#pragma unroll
    for (int u = 0; u < kPrefetch; ++u) {
      const int s = sb + u;
      if (s < ws1) {
        Slot& sl = slot[u];
        // activations for this step: B fragments
        const int kl = (s - cs0) * 32 + 8 * t;
        uint4 xb0 = make_uint4(0, 0, 0, 0), xb1 = make_uint4(0, 0, 0, 0);
        if (g < a.M) xb0 = *reinterpret_cast<const uint4*>(xs + g * a.xs_stride + kl);
        if (MT == 2 && g + 8 < a.M) xb1 = *reinterpret_cast<const uint4*>(xs + (g + 8) * a.xs_stride + kl);

        uint32_t P[4][4];
        if constexpr (FMT == EXQ_FMT_GPTQ4) {
          const int grp = s / a.gs_steps;
          if (grp != cur_grp) {
            cur_grp = grp;
            const uint32_t zs = sl.zw >> (4 * (col & 7));
#pragma unroll
            for (int c = 0; c < 4; ++c) gptq_zero_consts((zs >> (4 * c)) & 0xFu, zlo[c], zhi[c]);
            s2[0] = prmt(sl.sc.x, sl.sc.x, 0x1010);
            s2[1] = prmt(sl.sc.x, sl.sc.x, 0x3232);
            s2[2] = prmt(sl.sc.y, sl.sc.y, 0x1010);
            s2[3] = prmt(sl.sc.y, sl.sc.y, 0x3232);
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            unpack8_gptq(comp(sl.wa, c), zlo[c], zhi[c], P[c]);
#pragma unroll
            for (int i = 0; i < 4; ++i) P[c][i] = hmul2(P[c][i], s2[c]);
          }
        } else {
          s2[0] = prmt(sl.sc.x, sl.sc.x, 0x1010);
          s2[1] = prmt(sl.sc.x, sl.sc.x, 0x3232);
          s2[2] = prmt(sl.sc.y, sl.sc.y, 0x1010);
          s2[3] = prmt(sl.sc.y, sl.sc.y, 0x3232);
          switch (sl.bits) {
            case 2: exl2_cols<2>(sl, s2, P); break;
            case 3: exl2_cols<3>(sl, s2, P); break;
            case 4: exl2_cols<4>(sl, s2, P); break;
            case 5: exl2_cols<5>(sl, s2, P); break;
            case 6: exl2_cols<6>(sl, s2, P); break;
            case 8: exl2_cols<8>(sl, s2, P); break;
            default:
              bad = 1;
#pragma unroll
              for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int i = 0; i < 4; ++i) P[c][i] = 0u;
          }
        }

        // refill this slot before the tensor-core work
        if (s + kPrefetch < ws1) load_slot<FMT>(a, sl, s + kPrefetch, t, col, col_ok);

#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // 16-row slab of the step
            const uint32_t a0 = P[2 * nt][2 * h], a1 = P[2 * nt + 1][2 * h];
            const uint32_t a2 = P[2 * nt][2 * h + 1], a3 = P[2 * nt + 1][2 * h + 1];
            mma16816(acc[0][nt], a0, a1, a2, a3, h ? xb0.z : xb0.x, h ? xb0.w : xb0.y);
            if constexpr (MT == 2) mma16816(acc[1][nt], a0, a1, a2, a3, h ? xb1.z : xb1.x, h ? xb1.w : xb1.y);
          }
        }
      }
    }
  }
  if (bad) atomicOr(&g_gemv_err, kDevErrBadSegment);

  // ---- reduce: warps of the CTA, then CTAs of the cluster (rank order)
  __syncthreads();  // xs is dead from here on; reuse smem as fp32 partials
  float* red = reinterpret_cast<float*>(smem);
  constexpr int kElems = MT * 8 * 32;  // [m][column]
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int m0 = 8 * mt + 2 * t, c0 = 4 * g + 2 * nt;
      float* r = red + warp * kElems;
      r[m0 * 32 + c0] = acc[mt][nt][0];
      r[(m0 + 1) * 32 + c0] = acc[mt][nt][1];
      r[m0 * 32 + c0 + 1] = acc[mt][nt][2];
      r[(m0 + 1) * 32 + c0 + 1] = acc[mt][nt][3];
    }
  __syncthreads();
  for (int e = threadIdx.x; e < kElems; e += kThreads) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v += red[w * kElems + e];
    red[e] = v;
  }

  if (ncta > 1) {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  } else {
    __syncthreads();
  }

  // rank r finalises the elements e with e % ncta == r
  const uint32_t red_s = static_cast<uint32_t>(__cvta_generic_to_shared(red));
  for (int e = crank + ncta * threadIdx.x; e < a.M * 32; e += ncta * kThreads) {
    float v;
    if (ncta > 1) {
      v = 0.f;
      for (int r = 0; r < ncta; ++r) {
        uint32_t remote;
        float pv;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(red_s + 4u * e), "r"(r));
        asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(pv) : "r"(remote) : "memory");
        v += pv;
      }
    } else {
      v = red[e];
    }
    const int m = e >> 5, c = e & 31;
    const int n = strip * 32 + c;
    if (n < a.N) a.y[static_cast<size_t>(m) * a.N + n] = __half_as_ushort(__float2half_rn(v));
  }
  if (ncta > 1) {
    // keep this CTA's partials alive until every rank has read them
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
  }
}

using KernelFn = void (*)(GemvArgs);

template <int FMT, int MT, bool PERM>
KernelFn kernel_ptr() {
  return gemv_kernel<FMT, MT, PERM>;
}

KernelFn pick_kernel(int fmt, int mt, bool perm) {
  if (fmt == EXQ_FMT_GPTQ4) {
    if (mt == 1) return perm ? kernel_ptr<EXQ_FMT_GPTQ4, 1, true>() : kernel_ptr<EXQ_FMT_GPTQ4, 1, false>();
    return perm ? kernel_ptr<EXQ_FMT_GPTQ4, 2, true>() : kernel_ptr<EXQ_FMT_GPTQ4, 2, false>();
  }
  if (mt == 1) return perm ? kernel_ptr<EXQ_FMT_EXL2, 1, true>() : kernel_ptr<EXQ_FMT_EXL2, 1, false>();
  return perm ? kernel_ptr<EXQ_FMT_EXL2, 2, true>() : kernel_ptr<EXQ_FMT_EXL2, 2, false>();
}

int xs_stride_for(int k_len) {
  // rows at an odd multiple of 64 bytes apart: the 8 lanes of a quarter-warp
  // (two token rows x four 16-byte blocks) hit distinct banks
  return (k_len % 64 == 32) ? k_len : k_len + 32;
}

}  // namespace

exq_status launch_gemv(const exq_weight& w, const uint16_t* x, int M, uint16_t* y, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EXQ_ERR_CUDA;
  const DeviceInfo& di = device_info(dev);
  if (di.sm_count <= 0) return EXQ_ERR_CUDA;

  const int n_steps = w.K / 32;
  const int n_strips = (w.N + 31) / 32;
  const int mt = M <= 8 ? 1 : 2;
  const bool perm = w.perm != nullptr;
  KernelFn fn = pick_kernel(w.format, mt, perm);

  static std::once_flag attr_once[8];
  const int fidx = (w.format == EXQ_FMT_GPTQ4 ? 0 : 4) + (mt - 1) * 2 + (perm ? 1 : 0);
  std::call_once(attr_once[fidx], [&] {
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, di.max_smem_optin);
  });

  // choose the cluster size C (CTAs splitting K per 32-column strip): a small
  // cost model of waves x per-warp steps, plus a reduction term per rank
  int best_c = -1;
  double best_cost = 1e30;
  for (int c = 1; c <= 8; ++c) {
    const int cta_steps = (n_steps + c - 1) / c;
    if (c > 1 && (c - 1) * cta_steps >= n_steps) break;  // an empty rank
    const int k_len = cta_steps * 32;
    const size_t xs_bytes = static_cast<size_t>(M) * xs_stride_for(k_len) * 2;
    const size_t red_bytes = static_cast<size_t>(kWarps) * mt * 8 * 32 * 4;
    const size_t smem = std::max(xs_bytes, red_bytes);
    if (smem > static_cast<size_t>(di.max_smem_optin)) continue;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, kThreads, smem) != cudaSuccess || occ <= 0) continue;
    const double slots = static_cast<double>(di.sm_count) * occ;
    const double waves = std::ceil(static_cast<double>(n_strips) * c / slots);
    const double per_warp = std::ceil(static_cast<double>(cta_steps) / kWarps);
    const double cost = waves * (per_warp + 1.5 + 0.35 * c);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best_c = c;
    }
  }
  if (const char* env = std::getenv("EXQ_GEMV_CLUSTER")) {
    const int c = std::atoi(env);
    if (c >= 1 && c <= 8) best_c = c;
  }
  if (best_c < 0) return EXQ_ERR_UNSUPPORTED;

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
  args.n_steps = n_steps;
  args.gs_steps = w.format == EXQ_FMT_GPTQ4 ? w.group_size / 32 : 1;
  args.n_word_rows = w.n_word_rows;
  args.cta_steps = (n_steps + best_c - 1) / best_c;
  args.xs_stride = xs_stride_for(args.cta_steps * 32);
  const size_t smem = std::max(static_cast<size_t>(M) * args.xs_stride * 2,
                               static_cast<size_t>(kWarps) * mt * 8 * 32 * 4);

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(best_c, n_strips, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeClusterDimension;
  attrs[na].val.clusterDim.x = best_c;
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
