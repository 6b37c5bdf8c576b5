// Prefill-sized fused quantized matmul on the 5th-generation tensor cores:
//   y[M, N] = x[M, K] . dequant(Wq)[K, N], fp16 in, fp32 accumulate, fp16 out.
//
// The ExLlamaV2 blog post ("ExLlamaV2: The fastest inference engine for
// quantized Llama/HF models", section "How the Fused CUDA Kernel Works")
// describes the fused kernel as loading packed weights, dequantising on the
// fly and doing the matmul in the same kernel without an intermediate write,
// "using tensor cores". Here the product is computed transposed, y^T = W^T x^T,
// so that the dequantised weights are the MMA's A operand and live in tensor
// memory, never in shared memory. Per CTA tile of 128 output columns x 256
// tokens and per 64-row K slab:
//
//   warp 0      TMA producer: the x tile (256 tokens x 64 fp16, 128-byte
//               swizzle), the packed word rows of the slab as one tensor-map
//               box of 128 columns (8 rows for GPTQ; 16 rows for EXL2, the
//               most two segments take, so the box may run into the next
//               slab's rows: one copy per slab costs less than one per
//               segment), its scale rows and GPTQ zero rows, all completing
//               on one mbarrier per stage (5 stages).
//   warps 2-9   dequantisers: thread = output column (its TMEM lane), warp
//               pair = the slab's two 32-row halves; packed words -> exact
//               fp16 (q - z) -> * s, stored with tcgen05.st as the K-major A
//               operand (128 lanes x 32 columns per stage); then the epilogue.
//   warp 1      allocates tensor memory; one elected lane issues
//               tcgen05.mma.kind::f16 with A in TMEM and x (B, N = up to 256
//               tokens) in shared memory, M = 128, K = 16, four per slab,
//               accumulating fp32 in TMEM, and commits each stage back to its
//               "empty" mbarrier.
//   epilogue    tcgen05.ld 32x32b (lane = output column, column = token) ->
//               fp16 -> global; with a K split, fp32 partial sums go to the
//               workspace and a second kernel adds them in split order.
//
// Act-order (a stored-row permutation) is applied to x by a gather kernel
// into the caller's workspace first, so the tensor map reads x in stored-row
// order. Every mbarrier wait is bounded; on expiry the kernel records a
// timeout in its device error word, drains its own copies and frees TMEM.
#include <cuda.h>

#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "exq_device.cuh"
#include "exq_internal.h"

namespace exq {
namespace {

__device__ unsigned g_gemm_err;

constexpr int BN = 128;   // output columns per CTA = MMA M = TMEM lanes
constexpr int BT = 256;   // tokens per CTA = MMA N (at most)
constexpr int BK = 64;    // K rows per stage
constexpr int kStages = 5;
constexpr int kDequantWarps = 8;
constexpr int kThreads = (2 + kDequantWarps) * 32;

// per-stage shared memory layout (bytes)
constexpr int kXBytes = BT * BK * 2;        // 32 KB, 1024-aligned
constexpr int kPackedBytes = 16 * BN * 4;   // up to 16 word rows (two 8-bit segments)
__host__ __device__ constexpr int packed_rows(int fmt) { return fmt == EXQ_FMT_GPTQ4 ? 8 : 16; }
constexpr int kScaleBytes = 2 * BN * 2;     // two 32-row halves
constexpr int kZeroStride = 128;            // each half's zero row on its own 128-byte boundary (TMA)
constexpr int kZeroBytes = 2 * kZeroStride;
constexpr int kOffX = 0;
constexpr int kOffPacked = kOffX + kXBytes;
constexpr int kOffScale = kOffPacked + kPackedBytes;
constexpr int kOffZero = kOffScale + kScaleBytes;
constexpr int kStageBytes = ((kOffZero + kZeroBytes + 1023) / 1024) * 1024;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /* barriers */ + 1024 /* alignment */;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
// every TMA destination starts on a 128-byte boundary (1024 for the swizzled x tile)
static_assert(kOffX % 1024 == 0, "operand alignment");
static_assert(kOffPacked % 128 == 0 && (BN * 4) % 128 == 0, "packed-row boxes");
static_assert(kOffScale % 128 == 0 && (BN * 2) % 128 == 0, "scale boxes");
static_assert(kOffZero % 128 == 0 && (BN / 8) * 4 <= kZeroStride, "zero boxes");
static_assert(kStageBytes % 1024 == 0, "stage alignment");

// tensor memory: fp32 accumulator (128 lanes x BT columns), then one A stage
// (128 lanes x BK / 2 columns: two fp16 per 32-bit cell) per pipeline stage
constexpr uint32_t kTmemAcc = 0;
constexpr uint32_t kTmemA = BT;
constexpr uint32_t kAStageCols = BK / 2;
constexpr uint32_t kTmemCols = 512;
static_assert(kTmemA + kStages * kAStageCols <= kTmemCols, "tensor memory budget");
constexpr int kWaitLimit = 1 << 22;  // try_wait rounds before giving up

// K split of grids with few tiles: at most 8 splits, each of at least 8 slabs
constexpr int kMaxSplit = 8;
constexpr int kMinSlabsPerSplit = 8;
constexpr int kSplitSmBound = 256;  // SM count the workspace bound allows for

constexpr int kMaxLayers = EXQ_GEMM_MAX_LAYERS;  // layers of one launch (they share x and K)

struct GemmMaps {
  CUtensorMap x;                // activations [rows, K] fp16, boxes 64 x 256, 128-byte swizzle
  CUtensorMap w[kMaxLayers];    // qweight [rows, N] uint32, boxes 128 columns x 8 (GPTQ) or 16 (EXL2) rows
  CUtensorMap s[kMaxLayers];    // scales [groups, N] fp16, boxes 128 x 1 (unused with two-level scales)
  CUtensorMap z[kMaxLayers];    // GPTQ zeros or two-level scale codes [groups, N / 8] uint32, boxes 16 x 1
};

// One layer of a launch: its column tiles are the grid's y indices
// tile0 .. (next layer's tile0) - 1; unused entries have tile0 = INT_MAX.
struct GemmLayer {
  const uint32_t* seg_off;      // EXL2 [S + 1]
  const uint16_t* q_scale_max;  // EXL2 two-level column maxima [N]
  uint16_t* y;                  // [M, N]
  int N, n_word_rows;
  int tile0;
  int x_row;                    // first row of the layer's activations in the x map
};

struct GemmArgs {
  GemmLayer L[kMaxLayers];
  float* part;      // [split, M, N] fp32 partial sums when split > 1 (one layer only)
  int M, K, gs;
  int split;        // CTAs along K (gridDim.z)
  int slabs_per;    // 64-row slabs per split (the last split may have fewer)
  int wait_limit;   // polling rounds of a bounded wait (kWaitLimit unless a test lowers it)
  int starve;       // test hook: the producer issues nothing, so the other roles' waits run out
};

// the layer that owns column tile T (constant indices into the parameters)
__device__ __forceinline__ int gemm_layer_of(const GemmArgs& a, int T) {
  int L = 0;
#pragma unroll
  for (int i = 1; i < kMaxLayers; ++i) L += T >= a.L[i].tile0 ? 1 : 0;
  return L;
}

struct StageMeta {  // written by the producer before the stage's copies
  int rows0, rows1;  // word rows of the two 32-row halves (EXL2 widths; GPTQ 4, 4)
};

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// bounded wait; returns false (and records a timeout) if the phase never completes
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int limit) {
  for (int i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  atomicOr(&g_gemm_err, kDevErrTimeout);
  *abort_flag = 1;
  return false;
}

// Bounded wait by a whole warp: lane 0 polls and broadcasts, so the loop
// exits for all lanes in the same round and warp-collective instructions that
// follow (tcgen05.ld/st.sync.aligned, __syncwarp) are reached convergently.
// Bounded wait of a whole warp. VOTE: every lane tests, and the warp leaves
// when a vote says all saw the phase complete (it stays complete until this
// warp acts on it) or one saw the abort flag; otherwise lane 0 tests and
// broadcasts. With the vote (and the dequantisers' per-lane release) the
// EXL2 formats ran 9-18 % faster; for GPTQ the vote alone made the large
// shapes 1-2 % slower, so GPTQ keeps the lane-0 test.
template <bool VOTE>
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                               int limit) {
  const bool leader = (threadIdx.x & 31) == 0;
  for (int i = 0; i < limit; ++i) {
    if constexpr (VOTE) {
      if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
      if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
    } else {
      int state = 0;  // 1 = phase complete, 2 = another role gave up
      if (leader) state = mbar_try_wait(bar, parity) ? 1 : (*abort_flag ? 2 : 0);
      state = __shfl_sync(0xffffffffu, state, 0);
      if (state == 1) return true;
      if (state == 2) return false;
    }
  }
  if (leader) atomicOr(&g_gemm_err, kDevErrTimeout);
  *abort_flag = 1;
  return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFF) >> 4);        // start address
  d |= static_cast<uint64_t>(1) << 16;                        // leading byte offset (unused for SW128 K-major)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;                // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                        // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                        // swizzle: 128B
  return d;
}

// instruction descriptor: D fp32, A/B fp16, both K-major, M = 128 (= BN),
// N = n (a multiple of 16, at most 256)
__device__ __forceinline__ uint32_t idesc_for(int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(BN >> 4) << 24);
}

// D[tmem] (+)= A[tmem] . B[smem]^T: A (128 x 16 fp16) read from tensor memory
__device__ __forceinline__ void umma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(tmem_d), "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ bool valid_width(int b) {
  return b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8;
}

// 8 codes of one column, dequantised, in natural K order (k0, k1), ..., (k6, k7)
__device__ __forceinline__ uint4 natural_order(const uint32_t (&P)[4]) {
  uint4 o;
  o.x = prmt(P[0], P[1], 0x5410);
  o.y = prmt(P[2], P[3], 0x5410);
  o.z = prmt(P[0], P[1], 0x7632);
  o.w = prmt(P[2], P[3], 0x7632);
  return o;
}

// the same in the K order of the x tile: natural, or, when the gather stored
// x pair-interleaved (XP: k0 k4 k1 k5 k2 k6 k3 k7), the unpackers' pairs as
// they are
template <bool XP>
__device__ __forceinline__ uint4 k_order(const uint32_t (&P)[4]) {
  if constexpr (XP) return make_uint4(P[0], P[1], P[2], P[3]);
  return natural_order(P);
}

// QS: two-level scales, s2 = the exact fraction (c + 1) / 16 and m2 the
// column maximum (the first multiply is exact, the second is the rounding)
template <int B, bool XP, bool QS>
__device__ __forceinline__ uint4 exl2_block(const uint32_t* rows, int t, int col, uint32_t s2, uint32_t m2) {
  int wi, off;
  block_window(B, t, wi, off);
  const uint32_t wa = rows[wi * BN + col];
  const uint32_t wb = block_needs_second(B, off) ? rows[(wi + 1) * BN + col] : 0u;
  uint32_t P[4];
  unpack8<B>(fshr(wa, wb, off), wb >> off, P);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    P[i] = hmul2(P[i], s2);
    if constexpr (QS) P[i] = hmul2(P[i], m2);
  }
  return k_order<XP>(P);
}

// the 32 codes of one column of a width-B segment -> 16 registers of fp16
// pairs in K order (one TMEM A-operand row of the half slab)
template <int B, bool XP, bool QS>
__device__ __forceinline__ void exl2_segment(const uint32_t* rows, int col, uint32_t s2, uint32_t m2,
                                             uint32_t (&r)[16]) {
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint4 o = exl2_block<B, XP, QS>(rows, t, col, s2, m2);
    r[4 * t + 0] = o.x;
    r[4 * t + 1] = o.y;
    r[4 * t + 2] = o.z;
    r[4 * t + 3] = o.w;
  }
}

// ---------------------------------------------------------------- the kernel

template <int FMT, bool XP>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmArgs a) {
  constexpr bool kVote = FMT != EXQ_FMT_GPTQ4;  // the dequantisers' wait style (see mbar_wait_warp)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* bar_area = smem + kStages * kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(bar_area);
  uint64_t* aready = full + kStages;
  uint64_t* empty = aready + kStages;
  uint64_t* accum = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  StageMeta* meta = reinterpret_cast<StageMeta*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // token tiles vary fastest, so the CTAs that share a column tile's packed
  // weights run together and the repeats come from L2
  const int m0 = blockIdx.x * BT;
  const int layer = gemm_layer_of(a, blockIdx.y);
  const GemmLayer* ly = &a.L[0] + layer;  // read through the parameter block, no select chain
  const int n0 = (static_cast<int>(blockIdx.y) - ly->tile0) * BN;
  const int xm0 = ly->x_row + m0;         // the tile's first row in the x map
  const int kt0 = blockIdx.z * a.slabs_per;                      // this split's first slab
  const int n_iter = min(a.K / BK, kt0 + a.slabs_per) - kt0;     // >= 1 (host plan)
  const int tokens = min(BT, a.M - m0);                          // valid tokens of the tile
  const int n_mma = (tokens + 15) & ~15;                         // MMA N

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&aready[s]), kDequantWarps * 32);  // every lane of the dequantisers
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(accum), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !a.starve) {  // test hook: a starved producer issues nothing
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.x)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.w[0] + layer)) : "memory");
      int issued = 0;
      for (int i = 0; i < n_iter; ++i) {
        const int kt = kt0 + i;
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, abort_flag, a.wait_limit)) break;
        uint8_t* st = smem + s * kStageBytes;
        const uint32_t bar = smem_u32(&full[s]);
        int rows0, rows1;
        int row_start;
        if constexpr (FMT == EXQ_FMT_GPTQ4) {
          rows0 = rows1 = 4;
          row_start = kt * 8;
        } else {
          const unsigned o0 = __ldg(ly->seg_off + 2 * kt), o1 = __ldg(ly->seg_off + 2 * kt + 1),
                         o2 = __ldg(ly->seg_off + 2 * kt + 2);
          rows0 = static_cast<int>(o1 - o0);
          rows1 = static_cast<int>(o2 - o1);
          if (!valid_width(rows0) || !valid_width(rows1) || o2 > static_cast<unsigned>(ly->n_word_rows) ||
              o1 < o0) {
            atomicOr(&g_gemm_err, kDevErrBadSegment);
            rows0 = rows1 = 0;
          }
          row_start = static_cast<int>(o0);
        }
        meta[s].rows0 = rows0;
        meta[s].rows1 = rows1;
        const int rows = rows0 + rows1;
        // boxes always move their full size (rows past M and columns past N read as zero)
        uint32_t tx = kXBytes + (rows > 0 ? static_cast<uint32_t>(packed_rows(FMT)) * BN * 4u : 0u);
        if constexpr (FMT != EXQ_FMT_EXL2_QSCALE) tx += 2u * BN * 2u;  // fp16 scale rows
        if constexpr (FMT != EXQ_FMT_EXL2) tx += 2u * (BN / 8) * 4u;   // zero or scale-code rows
        mbar_expect_tx(bar, tx);
        tma_load_2d(smem_u32(st + kOffX), &maps.x, kt * BK, xm0, bar);
        if (rows > 0) tma_load_2d(smem_u32(st + kOffPacked), &maps.w[0] + layer, n0, row_start, bar);
        for (int h = 0; h < 2; ++h) {
          const int g = FMT == EXQ_FMT_GPTQ4 ? (kt * BK + 32 * h) / a.gs : 2 * kt + h;
          if constexpr (FMT != EXQ_FMT_EXL2_QSCALE)
            tma_load_2d(smem_u32(st + kOffScale + h * BN * 2), &maps.s[0] + layer, n0, g, bar);
          if constexpr (FMT != EXQ_FMT_EXL2)
            tma_load_2d(smem_u32(st + kOffZero + h * kZeroStride), &maps.z[0] + layer, n0 / 8, g, bar);
        }
        issued = i + 1;
      }
      // drain: every issued stage's copies must land before the CTA may exit
      for (int i = max(0, issued - kStages); i < issued; ++i) {
        const uint32_t bar = smem_u32(&full[i % kStages]);
        for (int r = 0; r < a.wait_limit; ++r)
          if (mbar_try_wait(bar, (i / kStages) & 1)) break;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_for(n_mma);
      for (int i = 0; i < n_iter; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!mbar_wait(smem_u32(&full[s]), ph, abort_flag, a.wait_limit)) break;
        if (!mbar_wait(smem_u32(&aready[s]), ph, abort_flag, a.wait_limit)) break;
        tc_fence_after();
        const uint64_t bdesc = sw128_desc(smem_u32(smem + s * kStageBytes + kOffX));
        const uint32_t a_tmem = tmem + kTmemA + s * kAStageCols;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)  // K = 16: 8 TMEM columns of A; +32 bytes of x = +2 encoded
          umma_f16_ts(tmem + kTmemAcc, a_tmem + 8 * k, bdesc + 2 * k, idesc, (i | k) != 0);
        umma_commit(smem_u32(&empty[s]));
      }
      umma_commit(smem_u32(accum));
    }
  } else {
    // ------------------------------------------------------------ dequantisers
    const int q = warp & 3;                      // the TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;               // its 32-row half of the slab
    const int col = q * 32 + lane;               // output column in the tile = A row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    // two-level scales: this column's fp16 maximum, in both halves
    uint32_t m2 = 0u;
    if constexpr (FMT == EXQ_FMT_EXL2_QSCALE) {
      const uint32_t m = __ldg(ly->q_scale_max + n0 + col);
      m2 = m | (m << 16);
    }
    for (int i = 0; i < n_iter; ++i) {
      const int s = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      if (!mbar_wait_warp<kVote>(smem_u32(&full[s]), ph, abort_flag, a.wait_limit)) break;
      if (!mbar_wait_warp<kVote>(smem_u32(&empty[s]), ph ^ 1, abort_flag, a.wait_limit)) break;  // A stage read by earlier MMAs
      tc_fence_after();
      const uint8_t* st = smem + s * kStageBytes;
      const uint32_t* packed = reinterpret_cast<const uint32_t*>(st + kOffPacked);
      uint32_t s2;
      if constexpr (FMT == EXQ_FMT_EXL2_QSCALE) {
        // the exact fraction (c + 1) / 16 of the column's 4-bit code; m2 follows
        const uint32_t cw = reinterpret_cast<const uint32_t*>(st + kOffZero + h * kZeroStride)[col >> 3];
        const uint32_t c = (cw >> (4 * (col & 7))) & 0xFu;
        s2 = two_level_frac2(c | (c << 16));
      } else {
        const uint16_t* sc = reinterpret_cast<const uint16_t*>(st + kOffScale);
        const uint32_t s16 = sc[h * BN + col];
        s2 = s16 | (s16 << 16);
      }
      uint32_t r[16];
      if constexpr (FMT == EXQ_FMT_GPTQ4) {
        const uint32_t zw = reinterpret_cast<const uint32_t*>(st + kOffZero + h * kZeroStride)[col >> 3];
        uint32_t zlo, zhi;
        gptq_zero_consts((zw >> (4 * (col & 7))) & 0xFu, zlo, zhi);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          uint32_t P[4];
          unpack8_gptq(packed[(4 * h + t) * BN + col], zlo, zhi, P);
#pragma unroll
          for (int j = 0; j < 4; ++j) P[j] = hmul2(P[j], s2);
          const uint4 o = k_order<XP>(P);
          r[4 * t + 0] = o.x;
          r[4 * t + 1] = o.y;
          r[4 * t + 2] = o.z;
          r[4 * t + 3] = o.w;
        }
      } else {
        const int b = h == 0 ? meta[s].rows0 : meta[s].rows1;
        const uint32_t* rows = packed + (h == 0 ? 0 : meta[s].rows0) * BN;
        // one branch per 32-row segment (warp-uniform), each width's 4 blocks unrolled inside
        switch (b) {
          case 2: exl2_segment<2, XP, FMT == EXQ_FMT_EXL2_QSCALE>(rows, col, s2, m2, r); break;
          case 3: exl2_segment<3, XP, FMT == EXQ_FMT_EXL2_QSCALE>(rows, col, s2, m2, r); break;
          case 4: exl2_segment<4, XP, FMT == EXQ_FMT_EXL2_QSCALE>(rows, col, s2, m2, r); break;
          case 5: exl2_segment<5, XP, FMT == EXQ_FMT_EXL2_QSCALE>(rows, col, s2, m2, r); break;
          case 6: exl2_segment<6, XP, FMT == EXQ_FMT_EXL2_QSCALE>(rows, col, s2, m2, r); break;
          case 8: exl2_segment<8, XP, FMT == EXQ_FMT_EXL2_QSCALE>(rows, col, s2, m2, r); break;
          default:
#pragma unroll
            for (int j = 0; j < 16; ++j) r[j] = 0u;
        }
      }
      tmem_st16(tmem + lane_base + kTmemA + s * kAStageCols + h * 16, r);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&aready[s]));  // each lane, its stores done
    }

    // ------------------------------------------------------------ epilogue
    // accumulator lane = output column, accumulator column = token; warp h
    // takes tokens [128 h, 128 h + 128) of its lane quarter
    if (mbar_wait_warp<kVote>(smem_u32(accum), 0, abort_flag, a.wait_limit) && !*abort_flag) {
      tc_fence_after();
      const int n = n0 + col;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        const int t0 = h * 128 + cc * 32;
        if (t0 >= tokens) break;  // warp-uniform
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kTmemAcc + t0, r);
        const int mt = tokens - t0;
        if (a.split == 1) {
          uint16_t* dst = ly->y + static_cast<size_t>(m0 + t0) * ly->N + n;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < mt) dst[static_cast<size_t>(j) * ly->N] = __half_as_ushort(__float2half_rn(__uint_as_float(r[j])));
        } else {
          float* dst = a.part + (static_cast<size_t>(blockIdx.z) * a.M + m0 + t0) * ly->N + n;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < mt) dst[static_cast<size_t>(j) * ly->N] = __uint_as_float(r[j]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// y = fp16(sum over splits of the fp32 partial sums), added in split order so
// the result does not depend on which CTA finished first. Launched as a
// programmatic dependent of the split GEMM.
__global__ void __launch_bounds__(256) split_reduce_kernel(const float* __restrict__ part, uint16_t* __restrict__ y,
                                                           long long mn, int split) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x * 8;
  for (long long e = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * 8; e < mn; e += stride) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    for (int z = 0; z < split; ++z) {
      const float4* p = reinterpret_cast<const float4*>(part + z * mn + e);
      const float4 u = __ldg(p), v = __ldg(p + 1);
      acc[0] += u.x; acc[1] += u.y; acc[2] += u.z; acc[3] += u.w;
      acc[4] += v.x; acc[5] += v.y; acc[6] += v.z; acc[7] += v.w;
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = __half_as_ushort(__float2half_rn(acc[2 * j])) |
             (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc[2 * j + 1]))) << 16);
    *reinterpret_cast<uint4*>(y + e) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// x_perm[l][m][j] = x[m][perm_l[j]]: act-order rows gathered once per layer of
// the launch (grid row l; a layer without a permutation gets a plain copy) so
// the tensor map reads activations in stored-row order. Entries outside
// [0, K) read as 0 and are reported.
struct PermArgs {
  const int32_t* perm[kMaxLayers];  // NULL: identity
};

__global__ void permute_x_kernel(const uint16_t* __restrict__ x, const __grid_constant__ PermArgs pa,
                                 uint16_t* __restrict__ xp, int M, int K, bool interleave) {
  const int l = blockIdx.y;
  const int32_t* perm = nullptr;
#pragma unroll
  for (int i = 0; i < kMaxLayers; ++i)
    if (l == i) perm = pa.perm[i];
  uint16_t* out = xp + static_cast<size_t>(l) * M * K;
  const int chunks = K / 8;
  const long long total = static_cast<long long>(M) * chunks;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(e / chunks), c = static_cast<int>(e % chunks);
    int p[8];
    if (perm) {
      const int4 p0 = __ldg(reinterpret_cast<const int4*>(perm + 8 * c));
      const int4 p1 = __ldg(reinterpret_cast<const int4*>(perm + 8 * c + 4));
      p[0] = p0.x; p[1] = p0.y; p[2] = p0.z; p[3] = p0.w;
      p[4] = p1.x; p[5] = p1.y; p[6] = p1.z; p[7] = p1.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) p[i] = 8 * c + i;
    }
    const uint16_t* xr = x + static_cast<size_t>(m) * K;
    uint32_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool ok = static_cast<unsigned>(p[i]) < static_cast<unsigned>(K);
      if (!ok) atomicOr(&g_gemm_err, kDevErrBadPerm);
      v[i] = ok ? __ldg(xr + p[i]) : 0u;
    }
    uint4 o;
    if (interleave) {  // k0 k4 k1 k5 k2 k6 k3 k7
      o = make_uint4(v[0] | (v[4] << 16), v[1] | (v[5] << 16), v[2] | (v[6] << 16), v[3] | (v[7] << 16));
    } else {
      o = make_uint4(v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16), v[6] | (v[7] << 16));
    }
    *reinterpret_cast<uint4*>(out + static_cast<size_t>(m) * K + 8 * c) = o;
  }
}

}  // namespace

namespace {

struct SplitPlan {
  int split;      // CTAs along K
  int slabs_per;  // 64-row slabs per split
};

// A grid of fewer than half an SM count of tiles is split along K: as many
// splits as fill the SMs, at most kMaxSplit, each of at least
// kMinSlabsPerSplit slabs, rounded so that no split is empty.
SplitPlan plan_split(int tiles, int slabs, int sms) {
  int s = 1;
  if (tiles * 2 <= sms) s = std::min(std::min(kMaxSplit, sms / tiles), slabs / kMinSlabsPerSplit);
  if (s < 1) s = 1;
  const int per = (slabs + s - 1) / s;
  return {(slabs + per - 1) / per, per};
}

// Activations gathered into each layer's stored-row order when any layer of
// the launch has a permutation: n * M * K * 2 bytes, rounded up to 256.
size_t gather_bytes(const exq_weight* w, int n, int M) {
  bool any = false;
  for (int i = 0; i < n; ++i) any = any || w[i].perm != nullptr;
  return any ? ((static_cast<size_t>(n) * M * w[0].K * 2 + 255) / 256) * 256 : 0;
}

size_t partial_bytes(const exq_weight& w, int M, int split) {
  return split > 1 ? static_cast<size_t>(split) * M * w.N * 4 : 0;
}

int tiles_of(const exq_weight& w, int M) { return (w.N / BN) * ((M + BT - 1) / BT); }

bool shapes_ok(const exq_weight* w, int n) {
  for (int i = 0; i < n; ++i)
    if (w[i].K % BK || w[i].N % BN) return false;
  return true;
}

bool encode(EncodeTiled enc, CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner,
            uint64_t outer, uint64_t stride, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  const cuuint64_t gdim[2] = {inner, outer};
  const cuuint64_t gstride[1] = {stride};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return enc(map, type, 2, const_cast<void*>(base), gdim, gstride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {

// Waves of one K-deep tile each (in units of one unsplit tile's time) that a
// launch of `tiles` CTAs split `split` ways along K takes on `sms` SMs: the
// CTAs are not persistent, so a partial last wave costs a whole one.
double launch_waves(int tiles, int split, int sms) {
  return static_cast<double>((static_cast<long long>(tiles) * split + sms - 1) / sms) / split;
}

// What a launch costs beyond its waves (start-up, pipeline fill, the K-split
// reduction), in the same units; ties go to fewer launches.
constexpr double kLaunchWaves = 0.15;

// The K split each layer of a group would take alone, within the workspace
// left after the gathered activations.
SplitPlan layer_plan(const exq_weight& w, int M, int sms, size_t room) {
  SplitPlan p = plan_split(tiles_of(w, M), w.K / BK, sms);
  if (p.split > 1 && partial_bytes(w, M, p.split) > room) p = {1, w.K / BK};
  return p;
}

// A group runs as one launch over its pooled tiles unless one launch per
// layer (each split as exq_gemm would split it) fills the SMs in fewer waves:
// q + k + v of a 70B model at M = 512 pools 160 tiles, two waves on 152 SMs,
// where q alone is one wave and k, v each an eighth of one split eight ways.
bool pool_layers(const exq_weight* w, int n, int M, int sms, size_t room) {
  if (n == 1) return false;
  int pooled = 0;
  double apart = kLaunchWaves * (n - 1);
  for (int i = 0; i < n; ++i) {
    pooled += tiles_of(w[i], M);
    const SplitPlan p = layer_plan(w[i], M, sms, room);
    apart += launch_waves(tiles_of(w[i], M), p.split, sms) + (p.split > 1 ? kLaunchWaves : 0.0);
  }
  return launch_waves(pooled, 1, sms) <= apart;
}

}  // namespace

// Gathered activations (act-order) plus the fp32 partial sums of the largest
// K split that any layer of the group takes alone on a device of up to
// kSplitSmBound SMs (layers launched one by one reuse one partial buffer);
// the launch plans for the actual device, which never needs more.
size_t gemm_workspace_bytes(const exq_weight* w, int n, int M) {
  size_t bytes = gather_bytes(w, n, M), part = 0;
  if (shapes_ok(w, n) && M >= 1)
    for (int i = 0; i < n; ++i)
      part = std::max(part, partial_bytes(w[i], M, plan_split(tiles_of(w[i], M), w[i].K / BK, kSplitSmBound).split));
  return bytes + part;
}

size_t gemm_gather_bytes(const exq_weight& w, int M) { return gather_bytes(&w, 1, M); }

namespace {

// One gemm_kernel launch over the pooled column tiles of layers w[0, n),
// reading x rows [x_row_i, x_row_i + M) of the [x_rows, K] activations `xa`
// (pair-interleaved when `xp_mode`); with plan.split > 1 (n == 1 only) the
// fp32 partials go to `part` and a reduction kernel writes y[0].
exq_status launch_tiles(EncodeTiled enc, const exq_weight* w, int n, const uint16_t* xa, bool xp_mode,
                        int x_rows, bool stacked, int M, uint16_t* const* y, SplitPlan plan, float* part, int sms,
                        cudaStream_t stream) {
  const exq_weight& w0 = w[0];
  GemmMaps maps;
  std::memset(&maps, 0, sizeof maps);
  if (!encode(enc, &maps.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xa, w0.K, static_cast<uint64_t>(x_rows),
              static_cast<uint64_t>(w0.K) * 2, BK, BT, CU_TENSOR_MAP_SWIZZLE_128B))
    return EXQ_ERR_CUDA;
  GemmArgs args{};
  int tiles = 0;
  for (int i = 0; i < kMaxLayers; ++i) {
    GemmLayer& l = args.L[i];
    if (i >= n) {
      l.tile0 = INT_MAX;
      continue;
    }
    const exq_weight& wi = w[i];
    if (!encode(enc, &maps.w[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, wi.qweight, wi.N, wi.n_word_rows,
                static_cast<uint64_t>(wi.N) * 4, BN, packed_rows(wi.format), CU_TENSOR_MAP_SWIZZLE_NONE))
      return EXQ_ERR_CUDA;
    if (wi.scales && !encode(enc, &maps.s[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, wi.scales, wi.N, wi.n_groups,
                             static_cast<uint64_t>(wi.N) * 2, BN, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
      return EXQ_ERR_CUDA;
    if (wi.format != EXQ_FMT_EXL2) {  // GPTQ zeros or two-level scale codes
      const uint32_t* zsrc = wi.format == EXQ_FMT_GPTQ4 ? wi.qzeros : wi.q_scale;
      if (!encode(enc, &maps.z[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, zsrc, wi.N / 8, wi.n_groups,
                  static_cast<uint64_t>(wi.N / 8) * 4, BN / 8, 1, CU_TENSOR_MAP_SWIZZLE_NONE))
        return EXQ_ERR_CUDA;
    }
    l.seg_off = wi.seg_word_off;
    l.q_scale_max = wi.q_scale_max;
    l.y = y[i];
    l.N = wi.N;
    l.n_word_rows = wi.n_word_rows;
    l.tile0 = tiles;
    l.x_row = stacked ? i * M : 0;
    tiles += wi.N / BN;
  }
  args.part = part;
  args.M = M;
  args.K = w0.K;
  args.gs = w0.group_size;
  args.split = plan.split;
  args.slabs_per = plan.slabs_per;
  const int starve = testing_starve_rounds();
  args.wait_limit = starve > 0 ? starve : kWaitLimit;
  args.starve = starve > 0 ? 1 : 0;

  auto fn = w0.format == EXQ_FMT_GPTQ4
                ? (xp_mode ? gemm_kernel<EXQ_FMT_GPTQ4, true> : gemm_kernel<EXQ_FMT_GPTQ4, false>)
            : w0.format == EXQ_FMT_EXL2
                ? (xp_mode ? gemm_kernel<EXQ_FMT_EXL2, true> : gemm_kernel<EXQ_FMT_EXL2, false>)
                : (xp_mode ? gemm_kernel<EXQ_FMT_EXL2_QSCALE, true> : gemm_kernel<EXQ_FMT_EXL2_QSCALE, false>);
  static std::once_flag attr_once[6];
  std::call_once(attr_once[2 * (w0.format - 1) + (xp_mode ? 1 : 0)],
                 [&] { cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes); });
  {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((M + BT - 1) / BT, tiles, plan.split);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    if (cudaLaunchKernelEx(&cfg, fn, maps, args) != cudaSuccess) return EXQ_ERR_CUDA;
  }

  if (plan.split > 1) {  // one layer
    const long long mn = static_cast<long long>(M) * w0.N;
    const long long vecs = mn / 8;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(std::min<long long>((vecs + 255) / 256, 8LL * sms)));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, split_reduce_kernel, static_cast<const float*>(part), y[0], mn, plan.split) !=
        cudaSuccess)
      return EXQ_ERR_CUDA;
  }
  return EXQ_OK;
}

}  // namespace

exq_status launch_gemm(const exq_weight* w, int n, const uint16_t* x, int M, uint16_t* const* y, void* workspace,
                       size_t ws_bytes, cudaStream_t stream) {
  if (n < 1 || n > kMaxLayers) return EXQ_ERR_INVALID_ARG;
  if (!shapes_ok(w, n)) return EXQ_ERR_UNSUPPORTED;
  EncodeTiled enc = tensor_map_encoder();
  if (!enc) return EXQ_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EXQ_ERR_CUDA;
  const int sms = std::min(device_info(dev).sm_count, kSplitSmBound);
  const int K = w[0].K;

  const size_t gbytes = gather_bytes(w, n, M);
  const size_t room = workspace && ws_bytes > gbytes ? ws_bytes - gbytes : 0;
  float* part = room ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + gbytes) : nullptr;

  // a permuted layer: x gathered once into every layer's stored-row order,
  // layer i's copy at rows [i * M, (i + 1) * M), pair-interleaved
  const bool gather = gbytes > 0;
  const uint16_t* xa = x;
  if (gather) {
    uint16_t* xp = static_cast<uint16_t*>(workspace);
    PermArgs pa{};
    for (int i = 0; i < n; ++i) pa.perm[i] = w[i].perm;
    const long long total = static_cast<long long>(M) * (K / 8);
    const int blocks = static_cast<int>(std::min<long long>((total + 255) / 256, 4096));
    permute_x_kernel<<<dim3(blocks, n), 256, 0, stream>>>(x, pa, xp, M, K, true);
    if (cudaGetLastError() != cudaSuccess) return EXQ_ERR_CUDA;
    xa = xp;
  }

  if (pool_layers(w, n, M, sms, room))
    return launch_tiles(enc, w, n, xa, gather, gather ? n * M : M, gather, M, y, SplitPlan{1, K / BK}, nullptr, sms,
                        stream);
  for (int i = 0; i < n; ++i) {
    const SplitPlan p = layer_plan(w[i], M, sms, room);
    const uint16_t* xi = gather ? xa + static_cast<size_t>(i) * M * K : x;
    const exq_status st = launch_tiles(enc, w + i, 1, xi, gather, M, false, M, y + i, p, p.split > 1 ? part : nullptr,
                                       sms, stream);
    if (st != EXQ_OK) return st;
  }
  return EXQ_OK;
}

namespace {

// Scratch of exq_gemm_noalloc: the gathered activations of an act-order
// layer, for callers that cannot pass a workspace. Reserved statically, so
// every GPU that loads the library holds it until the process exits.
__device__ __align__(256) uint8_t g_noalloc_scratch[EXQ_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on `dev`, looked up with that device
// current (in host code the symbol is only a host-side stand-in, never a
// device address) on the first call that succeeds, then kept. A failed
// lookup is not kept: the next call tries again. nullptr if it failed.
void* noalloc_scratch(int dev) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* ptr[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) == cudaSuccess)
      ptr[dev] = p;
    else
      cudaGetLastError();
  }
  return ptr[dev];
}

}  // namespace

exq_status launch_gemm_noalloc(const exq_weight& w, const uint16_t* x, int M, uint16_t* y, cudaStream_t stream) {
  const size_t need = gather_bytes(&w, 1, M);
  if (need > EXQ_NOALLOC_SCRATCH_BYTES) return EXQ_ERR_UNSUPPORTED;
  // the set-up runs on the device's first call whatever the layer, so that a
  // caller who makes one call before stream capture has done it
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EXQ_ERR_CUDA;
  void* scratch = noalloc_scratch(dev);
  if (!scratch) return EXQ_ERR_CUDA;
  return launch_gemm(&w, 1, x, M, &y, need ? scratch : nullptr, need, stream);
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
