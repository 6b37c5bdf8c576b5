// Decode-sized fused quantized matmul, 1 <= M <= 16:  y = x . dequant(Wq),
// for one layer or for up to four layers that read the same x in one launch.
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
//  * Work is the list of (248-column tile, 32-row segment) units, tile-major,
//    over all layers of the launch (their tiles numbered one after another).
//    Every CTA takes an equal contiguous share, so all SMs stream the same
//    number of bytes whatever N and K are. A share falls into pieces, one per
//    tile it touches. For M <= 8 a CTA has one consumer set (8 warps) and
//    two CTAs share an SM (a ring of two slots each), so that on each SM a
//    CTA of the next call can start while the other CTA still finishes this
//    one; for M <= 16 a CTA has two sets and owns its SM.
//  * The warp after the consumers is the producer. It cuts each piece into
//    stages of at most 32 packed word rows, 40 for EXL2 at small M (EXL2: the
//    longest run of whole segments that fits, at most 16, one compare per
//    lane on the segment table's prefix sums; GPTQ: 8-segment blocks aligned
//    to 256 rows) and moves a stage with tensor-map copies into one slot of a
//    shared-memory ring: the word rows (a 32- or 40-row x 248-column box), the scale rows (a 16 x 248 box) and the
//    stage's activations (one or two 256 x M boxes); GPTQ zero rows follow as
//    4-byte asynchronous copies. All of it completes on the slot's "full"
//    mbarrier. The weight copies of the first slots are issued before the
//    wait on the previous kernel (they are model state); x after it.
//  * The consumer warps form one or two sets of eight: stage i goes to set
//    i % sets, and warp w of the set owns columns 32 w .. 32 w + 31 of the
//    tile for every segment of the stage, so the fixed cost of a stage (wait, descriptor,
//    release) is paid once per up to 16 segments. Lane (g = lane / 4,
//    t = lane % 4) owns the four columns 4g .. 4g+3 (one 16-byte read per
//    word row: eight lanes read a whole line) and the 8-code block t of every
//    segment. The tile is 248 columns wide so that a word row takes 992 bytes
//    in shared memory: the four rows that the lanes t = 0..3 of one
//    quarter-warp read then start 6 bank groups apart, and their 16-byte
//    reads do not collide. Codes are planted in the mantissa of 1024
//    (0x6400 | code << p), the zero is taken off exactly in fp16 and each pair
//    is scaled once (w = fp16_RN((q - z) s), the definition: the result is x
//    times the rounded fp16 weights), then fed to mma.sync m16n8k16 (fp16 in,
//    fp32 accumulate) as the A operand of a swapped product (A = W^T,
//    B = x^T), into four independent accumulators. A stage whose EXL2
//    segments share one width runs a loop compiled for that width.
//  * A piece's last stage carries a flush mark; with two sets the producer
//    queues an empty stage with the mark for the other set right after it,
//    so both sets close every piece. On the mark each warp writes fp32 partial sums of its
//    32 columns to the caller's workspace; the warp that arrives last at its
//    (tile, column group) counter adds the tile's partials in piece order,
//    writes y and puts the counter back to zero. Deterministic, and no warp
//    ever waits on another CTA.
//  * An act-order layer's x is gathered into stored-row order by a small
//    kernel first (into the workspace), once per call rather than per CTA; it
//    stores each 8-block as x0 x4 x1 x5 x2 x6 x3 x7, so that the consumers
//    read the MMA's operand pairs directly.
//  * EXL2 with two-level scales: instead of the scale box, the stage's rows
//    of 4-bit scale codes follow as 4-byte asynchronous copies (like GPTQ
//    zeros) and the tile's fp16 column maxima as one 16-byte copy per lane;
//    the consumers multiply each pair by the exact fraction (c + 1) / 16 and
//    then by the maximum m, so w = fp16_RN((q - z) ((c + 1) / 16) m) takes
//    one rounding.
//  * Programmatic dependent launch: every kernel lets the next launch start
//    early; the GEMV's first weight copies do not wait for the previous
//    kernel, its activations and outputs do.
//  * Every mbarrier wait is bounded; on expiry the kernel records a timeout
//    in its device error word and the other roles stop at their next wait.
#include <algorithm>
#include <climits>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "exq_device.cuh"
#include "exq_internal.h"

namespace exq {
namespace {

__device__ unsigned g_gemv_err;

constexpr int kTN = 248;                 // columns per tile (992-byte rows: see above)
constexpr int kTP = 256;                 // columns per tile in the partial sums (8 warps x 32)
constexpr int kColGroups = 8;            // 32 columns each
// Consumer sets: stage i is read by set i % sets. The kernels for M <= 8
// (one 8-token block) have one set per CTA and run two CTAs per SM where a
// ring of two slots fits half an SM's shared memory, so that one CTA can
// start its next call while the other still finishes; those for M <= 16 have
// two sets in one CTA per SM.
__host__ __device__ constexpr int sets_of(int MT) { return MT == 1 ? 1 : 2; }
constexpr int kMaxSegs = 16;             // EXL2 segments per stage
constexpr int kGptqSegs = 8;             // GPTQ segments per stage (256 rows of K); segments per x box
// Packed word rows per stage (the weight box's height), a kernel parameter
// ROWS: 32 in general (GPTQ: 8 segments of 4 rows), 40 for EXL2 where two
// slots of that height and the segment tables still fit half an SM (M <= 4
// on the 70B shapes): the stage's fixed cost is then spread over a quarter
// more segments (1.1 % faster on the 70B stream). Every call that fits takes
// 40, small ones too: a stream that switched between 32-row launches (small
// shares) and 40-row ones was 1.8 % slower than either, since consecutive
// launches then ask for different shared-memory sizes.
constexpr int kRowsShort = 32;
constexpr int kRowsLong = 40;
constexpr int kScaleRows = 16;           // scale (and GPTQ zero) rows per stage
constexpr int kCounterBytes = 64 * 1024; // workspace counter region (zero between calls)
constexpr int kMaxStages = 6;
// Stages whose weight copies go out before the wait on the previous kernel
// (their x copies follow the wait). A CTA that starts early has them ready
// when x arrives; one that starts when the previous kernel is already done
// gets its first x sooner than after a whole ring of weight copies: 3 of 5
// measured 0.6 % faster on the 70B stream than the whole ring (2: 0.5 %,
// 1: 0.8 % slower).
constexpr int kPreWaitStages = 3;
// try_wait rounds before giving up. The producer polls (a round without a
// suspend hint returns after a short, hardware-chosen time): it must issue
// the next copy as soon as a slot frees. Consumers of a two-set CTA sleep in
// the wait, up to kWaitHintNs a round, so that a set waiting for data does
// not take issue slots from the set that is computing (1.2 % faster on the
// 70B stream than polling there); those of a one-set CTA poll.
constexpr int kWaitLimit = 1 << 24;
constexpr int kSleepLimit = 1 << 17;       // consumer rounds: at most 2.6 s
constexpr uint32_t kWaitHintNs = 20000;

// slot layout (bytes): word rows [ROWS] | scale rows | GPTQ zero rows | x [2][M][256]
constexpr int kRowBytes = kTN * 4;                         // 992
constexpr int kScaleRowBytes = kTN * 2;                    // 496
constexpr int kZeroRowBytes = 128;                         // 31 zero words of a tile, one row per group
constexpr int kXBox = 256;                                 // activations per x box (8 segments)
constexpr int kXBoxBytes = kXBox * 2;                      // per token
constexpr int kSlotW = 0;
__host__ __device__ constexpr int slot_s(int rows) { return kSlotW + rows * kRowBytes; }
__host__ __device__ constexpr int slot_z(int rows) {
  return ((slot_s(rows) + kScaleRows * kScaleRowBytes + 127) / 128) * 128;
}
__host__ __device__ constexpr int slot_x(int rows) { return slot_z(rows) + kScaleRows * kZeroRowBytes; }
static_assert(slot_s(kRowsShort) % 128 == 0 && slot_z(kRowsShort) % 128 == 0 && slot_x(kRowsShort) % 128 == 0 &&
                  slot_s(kRowsLong) % 128 == 0 && slot_z(kRowsLong) % 128 == 0 && slot_x(kRowsLong) % 128 == 0,
              "tensor-map destinations start on 128-byte boundaries");
static_assert(kTN % 8 == 0 && kTN / 8 <= 32, "a tile's zero words fit one warp");
static_assert(kMaxSegs <= 2 * kGptqSegs, "a stage's activations fit two x boxes");
static_assert(kGptqSegs * 4 == kRowsShort, "a GPTQ stage fills the short box");

__host__ __device__ constexpr int slot_bytes_for(int M, int rows) {
  return ((slot_x(rows) + 2 * M * kXBoxBytes + 1023) / 1024) * 1024;
}

constexpr int kMaxLayers = EXQ_GEMV_MAX_LAYERS;  // layers of one launch (they share x and K)

struct GemvMaps {
  CUtensorMap w[kMaxLayers];  // qweight [n_word_rows, N] uint32, box 248 x 32
  CUtensorMap s[kMaxLayers];  // scales [groups, N] fp16, box 248 x 16
  CUtensorMap x;              // activations [rows, K] fp16 (stored-row order), box 256 x M
};

// One layer of a launch. Its tiles are the global tiles tile0 .. (next
// layer's tile0) - 1; unused entries have tile0 = INT_MAX.
struct GemvLayer {
  const uint32_t* seg_off;  // EXL2 [S + 1]
  const uint32_t* qzeros;   // GPTQ [G, N / 8]
  const uint32_t* q_scale;  // EXL2 two-level codes [S, N / 8]
  const uint16_t* q_scale_max;  // EXL2 two-level column maxima [N]
  uint16_t* y;              // [M, N]
  int N;
  int n_word_rows;
  int tile0;
  int x_row;                // first row of the layer's activations in the x map
};

struct GemvArgs {
  GemvLayer L[kMaxLayers];
  uint32_t* counters;       // [n_tiles][8], zero between calls
  float* partials;          // [n_tiles][max_pieces][M][kTP]
  int K, M;
  int S;                    // segments (K / 32)
  int gs_seg;               // GPTQ group size in segments
  int G;                    // GPTQ groups
  int n_tiles;              // tiles of all layers
  int total;                // units = n_tiles * S
  int max_pieces;
  int stages;
  int slot_bytes;
  int off_bar;              // byte offset of the barriers, descriptors and tables
  int wait_limit;           // polling rounds of a bounded wait (kWaitLimit unless a test lowers it)
  int sleep_limit;          // sleeping rounds of a consumer's wait (kSleepLimit unless a test lowers it)
  int starve;               // test hook: the producer issues nothing, so the consumers' waits run out
};

// the layer that owns global tile T (constant indices into the parameters)
__device__ __forceinline__ int layer_of(const GemvArgs& a, int T) {
  int L = 0;
#pragma unroll
  for (int i = 1; i < kMaxLayers; ++i) L += T >= a.L[i].tile0 ? 1 : 0;
  return L;
}

__device__ __forceinline__ GemvLayer layer_params(const GemvArgs& a, int L) {
  GemvLayer r = a.L[0];
#pragma unroll
  for (int i = 1; i < kMaxLayers; ++i)
    if (L == i) r = a.L[i];
  return r;
}

// Stage descriptor, written by the producer before the slot's copies.
//   a: segments n (0..16) | flags
//   wlo, whi: EXL2 widths, 4 bits per segment (segments 0-7, 8-15; 0 = skip)
//   c: tile (global over the launch's layers) | layer << 16
//   gpos: GPTQ: position in its group of the stage's first segment
//   seq: the stage's index in the CTA's sequence (see stage_wait)
struct Desc {
  uint32_t a, wlo, whi, c;
  uint32_t gpos, seq, pad1, pad2;
};
constexpr uint32_t kDescLast = 1u << 8;     // after this stage the set flushes its partial sums
constexpr uint32_t kDescEnd = 1u << 9;      // no more stages for this set
constexpr uint32_t kDescUniform = 1u << 10; // EXL2: every segment of the stage has the same width

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

// try_wait that may suspend the thread until the phase completes, at most
// kWaitHintNs
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kWaitHintNs)
      : "memory");
  return ok != 0;
}

// Bounded wait of a whole warp: every lane polls, and the warp leaves when a
// vote says all lanes saw the phase complete (it stays complete until the
// waiting warp itself acts on it) or one saw the abort flag, so all lanes
// leave in the same round and no lane's result is broadcast from another.
// A timeout is recorded and raises the abort flag; a raised flag makes every
// other waiter give up too.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, int limit) {
  const bool leader = (threadIdx.x & 31) == 0;
  for (int i = 0; i < limit; ++i) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
  }
  if (leader) {
    atomicOr(&g_gemv_err, kDevErrTimeout);
    *abort_flag = 1;
  }
  return false;
}

// The wait of a consumer set for stage j of its slot. With two sets both use
// every slot in turn, so with an odd slot count a set's successive stages in
// one slot are two phases of its full barrier apart, and a parity wait alone also passes while the
// barrier is still short of the other set's stage in between (same parity
// two phases back). The descriptor closes that gap: the producer writes
// stage j's descriptor, with seq = j, only after the slot's previous stage
// was released, hence after it landed; once the descriptor shows j, the
// barrier is at stage j or past it and the parity wait is exact.
// SLEEP: the waiting warps suspend in try_wait (two sets per CTA: a set that
// waits then leaves the issue slots to the one that computes); otherwise
// they poll (one set per CTA: 0.5 % faster on the 70B stream than sleeping).
template <bool SLEEP>
__device__ __forceinline__ bool stage_wait(const uint32_t* seq, uint32_t j, uint32_t bar, uint32_t parity,
                                           volatile int* abort_flag, int limit) {
  const volatile uint32_t* vseq = seq;
  for (int i = 0; i < limit; ++i) {
    // every lane tests for itself (no broadcast from one lane); the warp goes
    // on once all lanes saw the stage: a completed phase stays completed, so
    // lanes that raced the completion agree in the next round
    const bool ready = *vseq == j && (SLEEP ? mbar_try_wait_sleep(bar, parity) : mbar_try_wait(bar, parity));
    if (__all_sync(0xffffffffu, ready)) return true;
    if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
  }
  if ((threadIdx.x & 31) == 0) {
    atomicOr(&g_gemv_err, kDevErrTimeout);
    *abort_flag = 1;
  }
  return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// 4-byte asynchronous copy; cp_async_arrive adds one pending arrival to
// `bar` at once and makes it when all of this thread's earlier cp.async
// copies have landed
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// shared-memory reads through plain pointers: ordered after the mbarrier
// waits (asm volatile with a memory clobber) and free to be scheduled
__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint2 lds64(const uint8_t* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ __forceinline__ uint32_t comp(const uint4& v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// ---------------------------------------------------------------- one segment
// Lane (g, t) holds, for its four columns c = 0..3, the exact fp16 pairs
// P[c][i] = (v_i - z, v_{i+4} - z) of the codes v_0..v_7 of block t. The MMA
// rows are the columns: tile 0 = columns 0 (row g) and 1 (row g + 8), tile 1
// = columns 2 and 3. Slab 0 takes pairs 0 and 1, slab 1 pairs 2 and 3; each
// (tile, slab) has its own accumulator, so the four MMAs of a segment do not
// wait on one another. The activations xb[mt] hold the matching pairs of
// token g (+ 8 mt).

template <int MT>
using Acc = float[MT][2][2][4];

template <int MT>
__device__ __forceinline__ void seg_mma(Acc<MT>& D, const uint32_t (&P)[4][4], const uint32_t (&xb)[MT][4]) {
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = 2 * h;
      mma16816(D[mt][h][0], P[c][0], P[c + 1][0], P[c][1], P[c + 1][1], xb[mt][0], xb[mt][1]);
      mma16816(D[mt][h][1], P[c][2], P[c + 1][2], P[c][3], P[c + 1][3], xb[mt][2], xb[mt][3]);
    }
  }
}

// EXL2 width B: `row` points at the lane's first word row of block t (the
// lane's four columns), `off` is the block's bit offset in it.
template <int B>
__device__ __forceinline__ void exl2_unpack(const uint8_t* row, uint32_t off, uint32_t (&P)[4][4]) {
  const uint4 wa = lds128(row);
  uint4 wb = make_uint4(0u, 0u, 0u, 0u);
  if constexpr (B == 3 || B == 5 || B == 6 || B == 8) wb = lds128(row + kRowBytes);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t a = comp(wa, c);
    uint32_t lo = a, hi = 0u;
    if constexpr (B == 2) {
      lo = a >> off;
    } else if constexpr (B == 8) {
      hi = comp(wb, c);
    } else if constexpr (B == 3 || B == 5 || B == 6) {
      const uint32_t b = comp(wb, c);
      lo = fshr(a, b, off);
      hi = b >> off;
    }
    unpack8<B>(lo, hi, P[c]);
  }
}

// The lane's four column scales from one 8-byte read of a scale row: s2[c]
// is the word that holds column c's scale, in its low half for even c and
// its high half for odd c (scale_pairs broadcasts the half it needs).
__device__ __forceinline__ void scales4(const uint8_t* p, uint32_t (&s2)[4]) {
  const uint2 v = lds64(p);
  s2[0] = s2[1] = v.x;
  s2[2] = s2[3] = v.y;
}

// two-level scales: the exact fractions (c + 1) / 16 of the lane's four
// columns, laid out like scales4's words; `codes` = their 4-bit codes in the
// low 16 bits
__device__ __forceinline__ void qfracs4(uint32_t codes, uint32_t (&s2)[4]) {
  const uint32_t lo = codes & 0xFFFFu, hi = lo >> 8;
  s2[0] = s2[1] = two_level_frac2(lo | (lo << 12));  // columns 0, 1
  s2[2] = s2[3] = two_level_frac2(hi | (hi << 12));  // columns 2, 3
}

__device__ __forceinline__ __half2 as_h2(uint32_t v) {
  __half2 h;
  memcpy(&h, &v, 4);
  return h;
}
__device__ __forceinline__ uint32_t as_u32(__half2 h) {
  uint32_t v;
  memcpy(&v, &h, 4);
  return v;
}

// column c's half of a scales4 / qfracs4 word in both halves: written with
// the half2 intrinsics, so that the compiler can take the half as an
// operand of the multiply instead of a separate permute
__device__ __forceinline__ __half2 col_half(uint32_t w, int c) {
  return (c & 1) ? __high2half2(as_h2(w)) : __low2half2(as_h2(w));
}

// w = fp16_RN((q - z) s) for the lane's four columns: one fp16 multiply per
// pair, round to nearest even. Two-level scales: s2 = the exact fractions,
// m2 = the column maxima; (q - z) (c + 1) / 16 is exact and the multiply by
// the maximum is the one rounding.
template <int FMT>
__device__ __forceinline__ void scale_pairs(uint32_t (&P)[4][4], const uint32_t (&s2)[4], const uint32_t (&m2)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const __half2 s = col_half(s2[c], c);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 w = __hmul2_rn(as_h2(P[c][i]), s);
      if constexpr (FMT == EXQ_FMT_EXL2_QSCALE) w = __hmul2_rn(w, col_half(m2[c], c));
      P[c][i] = as_u32(w);
    }
  }
}

template <int MT>
__device__ __forceinline__ void zero_acc(Acc<MT>& a) {
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) a[mt][h][k][i] = 0.f;
}

// the pairs (x0,x4),(x1,x5),(x2,x6),(x3,x7) of 8 consecutive activations
// (from natural order; with XP the gather already stored each 8-block as
// x0 x4 x1 x5 x2 x6 x3 x7, so the words are the pairs)
template <bool XP>
__device__ __forceinline__ void x_pairs(const uint8_t* p, uint32_t (&xb)[4]) {
  const uint4 v = lds128(p);
  if constexpr (XP) {
    xb[0] = v.x;
    xb[1] = v.y;
    xb[2] = v.z;
    xb[3] = v.w;
  } else {
    xb[0] = prmt(v.x, v.z, 0x5410);
    xb[1] = prmt(v.x, v.z, 0x7632);
    xb[2] = prmt(v.y, v.w, 0x5410);
    xb[3] = prmt(v.y, v.w, 0x7632);
  }
}

// activations of token tiles 0 (and 1) for one segment; dx = byte distance
// from the lane's token of tile 0 to its token of tile 1
template <int MT, bool XP>
__device__ __forceinline__ void load_x(const uint8_t* xp, int dx, uint32_t (&xb)[MT][4]) {
  x_pairs<XP>(xp, xb[0]);
  if constexpr (MT == 2) x_pairs<XP>(xp + dx, xb[1]);
}

// Lane t's 8-code block of a width-B segment starts at stream bit 8 B t:
// byte offset of its first word row (relative to the segment) and bit offset.
template <int B>
__device__ __forceinline__ int blk_row_bytes(int t) {
  return ((8 * B * t) >> 5) * kRowBytes;
}
template <int B>
__device__ __forceinline__ uint32_t blk_bit(int t) {
  return static_cast<uint32_t>((8 * B * t) & 31);
}

// ---------------------------------------------------------------- work split
// Units u = tile * S + segment; CTA c owns [c * total / G, (c + 1) * total / G).

__host__ __device__ __forceinline__ int share_begin(int c, int total, int G) {
  return static_cast<int>(static_cast<long long>(c) * total / G);
}
// the CTA that owns unit u
__host__ __device__ __forceinline__ int share_owner(int u, int total, int G) {
  return static_cast<int>((static_cast<long long>(u + 1) * G - 1) / total);
}

// Act-order gather for the layers of a launch: xp[l][m][j] = x[m][perm_l[j]]
// (stored-row order; a layer without a permutation gets a plain copy), one
// element per thread so that many loads are in flight, one grid row per
// layer. Out-of-range entries read as 0 and are reported. It also pulls the
// EXL2 segment tables (S + 1 entries each) into L2 for the GEMV that follows.
struct GatherArgs {
  const int32_t* perm[kMaxLayers];      // NULL: identity
  const uint32_t* seg_off[kMaxLayers];  // NULL: nothing to prefetch
};

__global__ void __launch_bounds__(256) gather_x_kernel(const uint16_t* __restrict__ x,
                                                       const __grid_constant__ GatherArgs ga, int M, int K,
                                                       uint16_t* __restrict__ xp, int S) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int l = blockIdx.y;
  const int32_t* perm = nullptr;
  const uint32_t* seg_off = nullptr;
#pragma unroll
  for (int i = 0; i < kMaxLayers; ++i)
    if (l == i) {
      perm = ga.perm[i];
      seg_off = ga.seg_off[i];
    }
  const int e = blockIdx.x * blockDim.x + threadIdx.x;  // element of the layer's [M, K]
  if (seg_off && e * 32 <= S) asm volatile("prefetch.global.L2 [%0];" ::"l"(seg_off + e * 32));
  const bool in = e < M * K;
  const int j = in ? e % K : 0;
  const int p = !in ? 0 : perm ? __ldg(perm + j) : j;  // the permutation is model state: read it before the wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!in) return;
  const bool ok = static_cast<unsigned>(p) < static_cast<unsigned>(K);
  if (!ok) atomicOr(&g_gemv_err, kDevErrBadPerm);
  // stored interleaved inside each 8-block: x0 x4 x1 x5 x2 x6 x3 x7 (K % 32 == 0, so blocks do not straddle rows)
  const int dst = (e & ~7) | ((e & 3) << 1) | ((e >> 2) & 1);
  xp[static_cast<size_t>(l) * M * K + dst] =
      ok ? __ldg(x + static_cast<size_t>(e / K) * K + p) : static_cast<uint16_t>(0);
}

__device__ __forceinline__ bool valid_width(int b) { return b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8; }

// ---------------------------------------------------------------- consumers of one stage
// Pointers of a consumer lane into one slot: wp = its columns of the first
// word row, sp = its four scales of the first scale row, xp = its activations
// of the first segment, cp = its scale codes (two-level) of the first segment.

// EXL2, every segment of width B: n segments from those pointers
template <int FMT, int B, int MT, bool XP>
__device__ __forceinline__ void run_uniform(const uint8_t* wp, const uint8_t* sp, const uint8_t* xp, int dx,
                                            int t, int n, const uint32_t (&m2)[4], const uint8_t* cp, int csh,
                                            Acc<MT>& acc) {
  const uint8_t* wrow = wp + blk_row_bytes<B>(t);
  const uint32_t off = blk_bit<B>(t);
#pragma unroll 2
  for (int j = 0; j < n; ++j) {
    uint32_t xb[MT][4], s2[4], P[4][4];
    load_x<MT, XP>(xp + 64 * j, dx, xb);
    if constexpr (FMT == EXQ_FMT_EXL2_QSCALE)
      qfracs4(lds32(cp + j * kZeroRowBytes) >> csh, s2);
    else
      scales4(sp + j * kScaleRowBytes, s2);
    exl2_unpack<B>(wrow + j * (B * kRowBytes), off, P);
    scale_pairs<FMT>(P, s2, m2);
    seg_mma<MT>(acc, P, xb);
  }
}

// EXL2, a whole stage of width B (ROWS / B segments, at most 16): the loop
// runs a compile-time count, so every address is an immediate offset
template <int FMT, int B, int MT, bool XP, int ROWS>
__device__ __forceinline__ void run_full(const uint8_t* wp, const uint8_t* sp, const uint8_t* xp, int xbox, int dx,
                                         int t, const uint32_t (&m2)[4], const uint8_t* cp, int csh, Acc<MT>& acc) {
  constexpr int kN = (ROWS / B) < 16 ? ROWS / B : 16;
  const uint8_t* wrow = wp + blk_row_bytes<B>(t);
  const uint32_t off = blk_bit<B>(t);
  const uint8_t* xq = xp + xbox - 64 * kGptqSegs;  // segments 8.. read the second x box
#pragma unroll
  for (int j = 0; j < kN; ++j) {
    uint32_t xb[MT][4], s2[4], P[4][4];
    load_x<MT, XP>((j < kGptqSegs ? xp : xq) + 64 * j, dx, xb);
    if constexpr (FMT == EXQ_FMT_EXL2_QSCALE)
      qfracs4(lds32(cp + j * kZeroRowBytes) >> csh, s2);
    else
      scales4(sp + j * kScaleRowBytes, s2);
    exl2_unpack<B>(wrow + j * (B * kRowBytes), off, P);
    scale_pairs<FMT>(P, s2, m2);
    seg_mma<MT>(acc, P, xb);
  }
}

// One EXL2 segment of width B, whole: its activations and scales, unpack,
// scale, multiply. Each width of a mixed stage runs its own copy of all of
// it, so that nothing after the width dispatch has to merge the per-width
// values into common registers.
template <int FMT, int B, int MT, bool XP>
__device__ __forceinline__ void exl2_segment(const uint8_t* row, const uint8_t* sp, const uint8_t* xp, int dx, int t,
                                             const uint32_t (&m2)[4], const uint8_t* cp, int csh, Acc<MT>& acc) {
  uint32_t xb[MT][4], s2[4], P[4][4];
  load_x<MT, XP>(xp, dx, xb);
  if constexpr (FMT == EXQ_FMT_EXL2_QSCALE)
    qfracs4(lds32(cp) >> csh, s2);
  else
    scales4(sp, s2);
  exl2_unpack<B>(row + blk_row_bytes<B>(t), blk_bit<B>(t), P);
  scale_pairs<FMT>(P, s2, m2);
  seg_mma<MT>(acc, P, xb);
}

// EXL2, widths from the descriptor (4 bits per segment): n segments of one x
// box; returns the word row after them. Width 0 is a segment the producer
// rejected (reported): it takes no rows.
template <int FMT, int MT, bool XP>
__device__ __forceinline__ const uint8_t* run_mixed(const uint8_t* row, const uint8_t* sp, const uint8_t* xp, int dx,
                                                    int t, int n, uint32_t widths, const uint32_t (&m2)[4],
                                                    const uint8_t* cp, int csh, Acc<MT>& acc) {
  for (int j = 0; j < n; ++j, widths >>= 4) {
    const uint8_t* sj = sp + j * kScaleRowBytes;
    const uint8_t* xj = xp + 64 * j;
    const uint8_t* cj = cp + j * kZeroRowBytes;
    switch (widths & 15u) {
      case 2: exl2_segment<FMT, 2, MT, XP>(row, sj, xj, dx, t, m2, cj, csh, acc); row += 2 * kRowBytes; break;
      case 3: exl2_segment<FMT, 3, MT, XP>(row, sj, xj, dx, t, m2, cj, csh, acc); row += 3 * kRowBytes; break;
      case 4: exl2_segment<FMT, 4, MT, XP>(row, sj, xj, dx, t, m2, cj, csh, acc); row += 4 * kRowBytes; break;
      case 5: exl2_segment<FMT, 5, MT, XP>(row, sj, xj, dx, t, m2, cj, csh, acc); row += 5 * kRowBytes; break;
      case 6: exl2_segment<FMT, 6, MT, XP>(row, sj, xj, dx, t, m2, cj, csh, acc); row += 6 * kRowBytes; break;
      case 8: exl2_segment<FMT, 8, MT, XP>(row, sj, xj, dx, t, m2, cj, csh, acc); row += 8 * kRowBytes; break;
      default: break;
    }
  }
  return row;
}

// ---------------------------------------------------------------- the kernel
// MT: 8-token blocks (1 for M <= 8, 2 for M <= 16).

template <int FMT, int MT, bool XP, int ROWS>
__global__ void __launch_bounds__((sets_of(MT) * kColGroups + 1) * 32, 3 - sets_of(MT))
    gemv_kernel(const __grid_constant__ GemvMaps maps, const __grid_constant__ GemvArgs a) {
  constexpr int sets = sets_of(MT);
  constexpr int kSlotS = slot_s(ROWS), kSlotZ = slot_z(ROWS), kSlotX = slot_x(ROWS);
  extern __shared__ uint8_t smem_raw[];
  // aligned by pointer arithmetic on the shared array, so that every access
  // through it stays a shared-memory access
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + a.off_bar);
  uint64_t* empty = full + kMaxStages;
  Desc* desc = reinterpret_cast<Desc*>(empty + kMaxStages);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(desc + kMaxStages);
  int* pend = const_cast<int*>(abort_flag) + 4;           // [kMaxStages] x copies held back (producer)
  uint32_t* tbl = reinterpret_cast<uint32_t*>(smem + a.off_bar + 512);  // EXL2 segment offsets [layers][S + 1]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kColGroups * 32);  // every lane of the stage's set
      desc[i].seq = ~0u;                            // no stage yet
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __syncthreads();

  const int G = static_cast<int>(gridDim.x);
  const int u0 = share_begin(blockIdx.x, a.total, G), u1 = share_begin(blockIdx.x + 1, a.total, G);

  if (warp == sets * kColGroups) {
    // ------------------------------------------------------------ producer
    if (a.starve) return;  // test hook: nothing is issued, nothing is in flight
    // the layers this CTA's share touches
    const int la = layer_of(a, u0 / a.S), lb = layer_of(a, (u1 - 1) / a.S);
    if (lane == 0) {
#pragma unroll
      for (int l = 0; l < kMaxLayers; ++l)
        if (l >= la && l <= lb) {
          asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.w[l])) : "memory");
          if constexpr (FMT != EXQ_FMT_EXL2_QSCALE)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.s[l])) : "memory");
        }
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.x)) : "memory");
    }
    if constexpr (FMT != EXQ_FMT_GPTQ4) {
      // the segment tables are model state: copy them before the wait
#pragma unroll
      for (int l = 0; l < kMaxLayers; ++l)
        if (l >= la && l <= lb)
          for (int i = lane; i <= a.S; i += 32) cp_async4(smem_u32(tbl + l * (a.S + 1) + i), a.L[l].seg_off + i);
      asm volatile("cp.async.wait_all;" ::: "memory");
      __syncwarp();
    }
    const uint32_t x_bytes = static_cast<uint32_t>(a.M) * kXBoxBytes;  // one x box
    // two-level scales arrive by cp.async, not in the transaction count
    const uint32_t tx_w = ROWS * kTN * 4 + (FMT == EXQ_FMT_EXL2_QSCALE ? 0 : kScaleRows * kTN * 2);
    int slot = 0, ephase = 0, issued = 0, npend = 0;
    // the piece's layer: its index, tensor maps, first row of x, GPTQ zeros
    const CUtensorMap* mw = &maps.w[0];
    const CUtensorMap* ms = &maps.s[0];
    int layer = 0, xrow = 0, nz = 0, ncols = 0;  // ncols: the tile's columns (two-level maxima)
    const uint32_t* qz = nullptr;                // GPTQ zeros or two-level scale codes
    const uint16_t* qmax = nullptr;
    bool waited = false, ok = true;
    auto x_copies = [&](int sl, int seg, int nx, int xr) {
      uint8_t* st = smem + sl * a.slot_bytes;
      for (int b = 0; b < nx; ++b)
        tma_load_2d(smem_u32(st + kSlotX + b * a.M * kXBoxBytes), &maps.x, seg * 32 + b * kXBox, xr,
                    smem_u32(&full[sl]));
    };
    auto release_x = [&]() {  // the activations may be read once the previous kernel is done
      asm volatile("griddepcontrol.wait;" ::: "memory");
      if (lane == 0)
        for (int i = 0; i < npend; ++i)
          x_copies(pend[i] & 0x7F, (pend[i] >> 8) & 0xFFFF, (pend[i] & 0x80) ? 2 : 1,
                   static_cast<int>(static_cast<unsigned>(pend[i]) >> 24));
      npend = 0;
      waited = true;
    };
    auto next_slot = [&]() {
      ++issued;
      if (++slot == a.stages) {
        slot = 0;
        ephase ^= 1;
      }
    };
    // one stage into the next slot; false once a wait gave up
    // tile: global (for the consumers), lt: in the layer (for the copies)
    auto issue = [&](uint32_t da, uint32_t wlo, uint32_t whi, uint32_t gpos, int tile, int lt, int seg, int n,
                     int row0, int srow, int zrows, bool bad) -> bool {
      if (!waited && issued >= min(a.stages, kPreWaitStages)) release_x();
      if (!warp_wait(smem_u32(&empty[slot]), ephase ^ 1, abort_flag, a.wait_limit)) return false;
      uint8_t* st = smem + slot * a.slot_bytes;
      const uint32_t fb = smem_u32(&full[slot]);
      if (lane == 0)
        desc[slot] = Desc{da, wlo, whi, static_cast<uint32_t>(tile) | (static_cast<uint32_t>(layer) << 16), gpos,
                          static_cast<uint32_t>(issued), 0u, 0u};
      const int nx = n > kGptqSegs ? 2 : 1;
      if constexpr (FMT != EXQ_FMT_EXL2) {
        if (!bad) {
          // GPTQ zero rows or two-level scale-code rows: [rows, N / 8] words
          const int cw = lt * (kTN / 8) + lane;
          for (int r = 0; r < zrows; ++r)
            if (cw < nz && lane < kTN / 8)
              cp_async4(smem_u32(st + kSlotZ + r * kZeroRowBytes + lane * 4),
                        qz + static_cast<size_t>(srow + r) * nz + cw);
          // two-level: the tile's column maxima, 8 columns (16 bytes) per lane
          if constexpr (FMT == EXQ_FMT_EXL2_QSCALE)
            if (8 * lane < ncols) cp_async16(smem_u32(st + kSlotS + 16 * lane), qmax + lt * kTN + 8 * lane);
          cp_async_arrive(fb);  // one more pending arrival, made when this lane's copies land
        }
      }
      __syncwarp();
      if (lane == 0) {
        if (bad) {
          mbar_arrive(fb);
        } else {
          mbar_expect_tx(fb, tx_w + nx * x_bytes);
          tma_load_2d(smem_u32(st + kSlotW), mw, lt * kTN, row0, fb);
          if constexpr (FMT != EXQ_FMT_EXL2_QSCALE) tma_load_2d(smem_u32(st + kSlotS), ms, lt * kTN, srow, fb);
          if (waited) x_copies(slot, seg, nx, xrow);
        }
      }
      if (!bad && !waited) pend[npend++] = slot | (nx == 2 ? 0x80 : 0) | (seg << 8) | (xrow << 24);
      next_slot();
      return true;
    };
    // a stage without data: only its descriptor (a flush mark, with the
    // piece's tile and layer, or an end mark)
    auto mark = [&](uint32_t da, uint32_t dc) -> bool {
      if (!waited && issued >= min(a.stages, kPreWaitStages)) release_x();
      if (!warp_wait(smem_u32(&empty[slot]), ephase ^ 1, abort_flag, a.wait_limit)) return false;
      if (lane == 0) {
        desc[slot] = Desc{da, 0u, 0u, dc, 0u, static_cast<uint32_t>(issued), 0u, 0u};
        mbar_arrive(smem_u32(&full[slot]));
      }
      next_slot();
      return true;
    };

    for (int u = u0; u < u1 && ok;) {
      const int tile = u / a.S;
      layer = layer_of(a, tile);
      const GemvLayer ly = layer_params(a, layer);
      const int lt = tile - ly.tile0;
      mw = &maps.w[layer];
      ms = &maps.s[layer];
      xrow = ly.x_row;
      qz = FMT == EXQ_FMT_EXL2_QSCALE ? ly.q_scale : ly.qzeros;
      qmax = ly.q_scale_max;
      nz = ly.N / 8;
      ncols = min(kTN, ly.N - lt * kTN);
      const int sa = u - tile * a.S;
      const int sb = min(a.S, sa + (u1 - u));
      u += sb - sa;
      for (int seg = sa; seg < sb && ok;) {
        int n, row0, srow, zrows = 0;
        uint32_t wlo = 0, whi = 0, gpos = 0;
        bool bad = false, uniform = false;
        if constexpr (FMT == EXQ_FMT_GPTQ4) {
          n = min(sb, (seg / kGptqSegs + 1) * kGptqSegs) - seg;
          row0 = 4 * seg;
          srow = seg / a.gs_seg;
          gpos = static_cast<uint32_t>(seg - srow * a.gs_seg);
          zrows = (seg + n - 1) / a.gs_seg - srow + 1;
        } else {
          // the longest run of valid segments from seg (at most sixteen) whose
          // widths add up to at most ROWS rows, straight from the word-row prefix
          // sums: lane j tests segment seg + j
          const int sk = seg + lane;
          const bool cand = lane < kMaxSegs && sk < sb;
          const uint32_t* ltbl = tbl + layer * (a.S + 1);
          const uint32_t base = ltbl[seg];
          const uint32_t e0 = cand ? ltbl[sk] : 0u, e1 = cand ? ltbl[sk + 1] : 0u;
          const int b = static_cast<int>(e1) - static_cast<int>(e0);
          const bool good = cand && valid_width(b) && e1 <= static_cast<uint32_t>(ly.n_word_rows) &&
                            static_cast<int>(e1 - base) <= ROWS;
          const unsigned stop = __ballot_sync(0xffffffffu, !good);
          n = __ffs(stop) - 1;  // leading lanes that fit (stop always has a bit at or below lane 16)
          wlo = __reduce_or_sync(0xffffffffu, lane < n && lane < 8 ? static_cast<uint32_t>(b) << (4 * lane) : 0u);
          whi = __reduce_or_sync(0xffffffffu,
                                 lane < n && lane >= 8 ? static_cast<uint32_t>(b) << (4 * (lane - 8)) : 0u);
          row0 = static_cast<int>(base);
          srow = seg;
          zrows = n;
          if (n == 0) {  // the segment at seg itself is malformed: skip it alone, reported
            bad = true;
            n = 1;
            if (lane == 0) atomicOr(&g_gemv_err, kDevErrBadSegment);
          } else {
            const uint32_t rep = (wlo & 15u) * 0x11111111u;
            const uint32_t mlo = n >= 8 ? ~0u : (1u << (4 * n)) - 1u;
            const uint32_t mhi = n <= 8 ? 0u : n >= 16 ? ~0u : (1u << (4 * (n - 8))) - 1u;
            uniform = ((wlo ^ rep) & mlo) == 0 && ((whi ^ rep) & mhi) == 0;
          }
        }
        const bool last = seg + n == sb;
        const uint32_t da = static_cast<uint32_t>(n) | (last ? kDescLast : 0u) | (uniform ? kDescUniform : 0u);
        ok = issue(da, wlo, whi, gpos, tile, lt, seg, n, row0, srow, zrows, bad);
        seg += n;
      }
      // the other set closes the piece too
      if (sets == 2 && ok) ok = mark(kDescLast, static_cast<uint32_t>(tile) | (static_cast<uint32_t>(layer) << 16));
    }
    if (!waited) release_x();
    // one end mark per set
    const bool ended = ok && mark(kDescEnd, 0u) && (sets == 1 || mark(kDescEnd, 0u));
    // after a give-up no consumer will wait for the copies still in flight:
    // they land before the CTA may exit (otherwise the consumers saw them all)
    if (!ended && lane == 0)
      for (int i = max(0, issued - a.stages); i < issued; ++i) {
        const uint32_t bar = smem_u32(&full[i % a.stages]);
        for (int r = 0; r < a.wait_limit; ++r)
          if (mbar_try_wait(bar, (i / a.stages) & 1)) break;
      }
    asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }

  // -------------------------------------------------------------- consumers
  asm volatile("griddepcontrol.wait;" ::: "memory");  // y and the workspace are shared with earlier kernels
  const int g = lane >> 2, t = lane & 3;
  const int set = warp / kColGroups;
  const int w = warp % kColGroups;         // column group: columns 32w .. 32w+31 of the tile
  const int tok0 = min(g, a.M - 1), tok1 = min(g + 8, a.M - 1);
  const int lw = kSlotW + 128 * w + 16 * g;                   // the lane's columns in a word row
  const int ls = kSlotS + 64 * w + 8 * g;                     // its four scales in a scale row
  const int lx = kSlotX + tok0 * kXBoxBytes + 16 * t;         // its block of x, token tile 0
  const int dx = (tok1 - tok0) * kXBoxBytes;                  // to token tile 1
  const int xbox = a.M * kXBoxBytes;                          // to the second x box
  const int lc = kSlotZ + (4 * w + (g >> 1)) * 4;             // its zero word (GPTQ) / scale codes (two-level)
  const int csh = 16 * (g & 1);                               // its nibbles in that word
  Acc<MT> acc;
  zero_acc<MT>(acc);
  int slot = set, fphase = 0;  // this set's first stage (stages >= 2)
  for (uint32_t j = static_cast<uint32_t>(set);; j += sets) {
    if (!stage_wait<(sets > 1)>(&desc[slot].seq, j, smem_u32(&full[slot]), fphase, abort_flag,
                                sets > 1 ? a.sleep_limit : a.wait_limit))
      break;
    const Desc d = desc[slot];
    if (d.a & kDescEnd) break;
    const uint8_t* sl = smem + slot * a.slot_bytes;
    const int n = static_cast<int>(d.a & 31u);
    if constexpr (FMT != EXQ_FMT_GPTQ4) {
      // two-level: the lane's four column maxima (the same for every segment of the tile)
      uint32_t m2[4] = {0u, 0u, 0u, 0u};
      if constexpr (FMT == EXQ_FMT_EXL2_QSCALE) scales4(sl + ls, m2);
      const int n0 = min(n, kGptqSegs);
      if (d.a & kDescUniform) {
        auto uni = [&](auto width) {
          constexpr int B = decltype(width)::value;
          if (n == ((ROWS / B) < 16 ? ROWS / B : 16)) {
            run_full<FMT, B, MT, XP, ROWS>(sl + lw, sl + ls, sl + lx, xbox, dx, t, m2, sl + lc, csh, acc);
            return;
          }
          run_uniform<FMT, B, MT, XP>(sl + lw, sl + ls, sl + lx, dx, t, n0, m2, sl + lc, csh, acc);
          if (n > kGptqSegs)
            run_uniform<FMT, B, MT, XP>(sl + lw + kGptqSegs * B * kRowBytes, sl + ls + kGptqSegs * kScaleRowBytes,
                                        sl + lx + xbox, dx, t, n - kGptqSegs, m2,
                                        sl + lc + kGptqSegs * kZeroRowBytes, csh, acc);
        };
        switch (d.wlo & 15u) {
          case 2: uni(std::integral_constant<int, 2>{}); break;
          case 3: uni(std::integral_constant<int, 3>{}); break;
          case 4: uni(std::integral_constant<int, 4>{}); break;
          case 5: uni(std::integral_constant<int, 5>{}); break;
          case 6: uni(std::integral_constant<int, 6>{}); break;
          default: uni(std::integral_constant<int, 8>{}); break;
        }
      } else {
        const uint8_t* row =
            run_mixed<FMT, MT, XP>(sl + lw, sl + ls, sl + lx, dx, t, n0, d.wlo, m2, sl + lc, csh, acc);
        if (n > kGptqSegs)
          run_mixed<FMT, MT, XP>(row, sl + ls + kGptqSegs * kScaleRowBytes, sl + lx + xbox, dx, t, n - kGptqSegs,
                                 d.whi, m2, sl + lc + kGptqSegs * kZeroRowBytes, csh, acc);
      }
    } else {
      if (n == kGptqSegs && a.gs_seg == 4 && d.gpos == 0) {
        // a whole stage of two 128-row groups: every address is a
        // compile-time offset and the group change needs no test
#pragma unroll
        for (int j = 0; j < kGptqSegs; ++j) {
          uint32_t zlo[4], zhi[4], s2[4];
          const uint32_t zw = lds32(sl + lc + (j / 4) * kZeroRowBytes) >> csh;
#pragma unroll
          for (int c = 0; c < 4; ++c) gptq_zero_consts((zw >> (4 * c)) & 0xFu, zlo[c], zhi[c]);
          scales4(sl + ls + (j / 4) * kScaleRowBytes, s2);
          uint32_t xb[MT][4];
          load_x<MT, XP>(sl + lx + 64 * j, dx, xb);
          const uint4 wq = lds128(sl + lw + t * kRowBytes + j * 4 * kRowBytes);
          uint32_t P[4][4];
#pragma unroll
          for (int c = 0; c < 4; ++c) unpack8_gptq(comp(wq, c), zlo[c], zhi[c], P[c]);
          scale_pairs<FMT>(P, s2, s2);
          seg_mma<MT>(acc, P, xb);
        }
      } else {
        int rem = static_cast<int>(d.gpos);  // position of the stage's first segment in its group
        const uint8_t* zr = sl + lc;         // zero word of the current group
        const uint8_t* sr = sl + ls;         // scales of the current group
        const uint8_t* wr = sl + lw + t * kRowBytes;
        const uint8_t* xr = sl + lx;
        uint32_t zlo[4], zhi[4], s2[4];
        for (int j = 0; j < n; ++j) {
          if (j == 0 || rem == 0) {  // this stage's first segment, or a new group
            const uint32_t zw = lds32(zr) >> csh;
#pragma unroll
            for (int c = 0; c < 4; ++c) gptq_zero_consts((zw >> (4 * c)) & 0xFu, zlo[c], zhi[c]);
            scales4(sr, s2);
          }
          uint32_t xb[MT][4];
          load_x<MT, XP>(xr, dx, xb);
          const uint4 wq = lds128(wr);
          uint32_t P[4][4];
#pragma unroll
          for (int c = 0; c < 4; ++c) unpack8_gptq(comp(wq, c), zlo[c], zhi[c], P[c]);
          scale_pairs<FMT>(P, s2, s2);
          seg_mma<MT>(acc, P, xb);
          wr += 4 * kRowBytes;
          xr += 64;
          if (++rem == a.gs_seg) {
            rem = 0;
            zr += kZeroRowBytes;
            sr += kScaleRowBytes;
          }
        }
      }
    }
    mbar_arrive(smem_u32(&empty[slot]));  // each lane, once its reads of the slot are done
    slot += sets;
    if (slot >= a.stages) {
      slot -= a.stages;
      fphase ^= 1;
    }

    if (d.a & kDescLast) {
      // ---- this warp's share of the piece: 32 columns, one set. Every
      // (piece, set) leaves fp32 partial sums; the last of the tile's 2P
      // arrivals at the column group's counter adds them in order.
      const int tile = static_cast<int>(d.c & 0xFFFFu);
      const int first = share_owner(tile * a.S, a.total, G);
      const int P2 = sets * (share_owner(tile * a.S + a.S - 1, a.total, G) - first + 1);
      const int pslot = sets * (static_cast<int>(blockIdx.x) - first) + set;
      float* part = a.partials + (static_cast<size_t>(tile) * a.max_pieces + pslot) * a.M * kTP;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int m = 8 * mt + 2 * t + hh;
          if (m < a.M)
            *reinterpret_cast<float4*>(part + m * kTP + 32 * w + 4 * g) =
                make_float4(acc[mt][0][0][hh] + acc[mt][0][1][hh], acc[mt][0][0][2 + hh] + acc[mt][0][1][2 + hh],
                            acc[mt][1][0][hh] + acc[mt][1][1][hh], acc[mt][1][0][2 + hh] + acc[mt][1][1][2 + hh]);
        }
      zero_acc<MT>(acc);
      // the warp's stores, then one acquire-release increment by lane 0: it
      // publishes them and, for the last arriver, makes every other piece's
      // stores visible to the reads below
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        unsigned* ctr = a.counters + tile * kColGroups + w;
        unsigned old;
        asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(old) : "l"(ctr) : "memory");
        last = old == static_cast<unsigned>(P2 - 1);
        if (last) atomicExch(ctr, 0u);  // ready for the next call
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      __syncwarp();
      if (last) {
        const GemvLayer* lp = &a.L[0] + (d.c >> 16);
        const float* base = a.partials + static_cast<size_t>(tile) * a.max_pieces * a.M * kTP + 32 * w + lane;
        const int ncol = (tile - lp->tile0) * kTN + 32 * w + lane;
        const bool n_ok = 32 * w + lane < kTN && ncol < lp->N;
        const size_t stride = static_cast<size_t>(a.M) * kTP;
        for (int m = 0; m < a.M; ++m) {
          // pieces added in piece order, 32 loads in flight at a time
          const float* pm = base + static_cast<size_t>(m) * kTP;
          float v = 0.f;
          for (int p0 = 0; p0 < P2; p0 += 32) {
            float q[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) q[i] = p0 + i < P2 ? __ldcg(pm + (p0 + i) * stride) : 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) v += q[i];
          }
          if (n_ok) lp->y[static_cast<size_t>(m) * lp->N + ncol] = __half_as_ushort(__float2half_rn(v));
        }
      }
    }
  }
}

}  // namespace
}  // namespace exq

// ================================================================ host side

namespace exq {
namespace {

using KernelFn = void (*)(GemvMaps, GemvArgs);

// long: 40-row stages (EXL2 formats, M <= 8 kernels only)
template <int FMT, bool XP>
KernelFn pick_for(int M, bool long_rows) {
  if constexpr (FMT == EXQ_FMT_GPTQ4)
    return M <= 8 ? gemv_kernel<FMT, 1, XP, kRowsShort> : gemv_kernel<FMT, 2, XP, kRowsShort>;
  else
    return M > 8 ? gemv_kernel<FMT, 2, XP, kRowsShort>
           : long_rows ? gemv_kernel<FMT, 1, XP, kRowsLong> : gemv_kernel<FMT, 1, XP, kRowsShort>;
}

// XP: x comes from the gather kernel, pair-interleaved
template <bool XP>
KernelFn pick_fmt(int fmt, int M, bool long_rows) {
  return fmt == EXQ_FMT_GPTQ4 ? pick_for<EXQ_FMT_GPTQ4, XP>(M, long_rows)
         : fmt == EXQ_FMT_EXL2 ? pick_for<EXQ_FMT_EXL2, XP>(M, long_rows)
                               : pick_for<EXQ_FMT_EXL2_QSCALE, XP>(M, long_rows);
}

KernelFn pick_kernel(int fmt, int M, bool xp, bool long_rows) {
  return xp ? pick_fmt<true>(fmt, M, long_rows) : pick_fmt<false>(fmt, M, long_rows);
}

int variant_index(int fmt, int M, bool xp, bool long_rows) {
  return 8 * (fmt - 1) + 4 * (xp ? 1 : 0) + 2 * (long_rows ? 1 : 0) + (M <= 8 ? 0 : 1);
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

constexpr int kSmemPerCta = 227 * 1024;  // one CTA per SM (the sm_103 per-block maximum)
constexpr int kSmemHalf = 113 * 1024;    // two CTAs per SM (each also takes 1 KB the system reserves)

struct Plan {
  int G, S, n_tiles, total, max_pieces, stages, slot_bytes, off_bar;
  int rows;                   // word rows per stage (kRowsShort or kRowsLong)
  int sets;                   // consumer sets per CTA: sets_of(MT) of the kernel for M
  int per_sm;                 // CTAs per SM: 2 when two one-set CTAs fit an SM
  int tile0[kMaxLayers + 1];  // first global tile of each layer; tile0[n] = n_tiles
  bool gather;                // some layer has a permutation: x is gathered per layer
  size_t smem;                // dynamic shared memory bytes (with the alignment slack)
  size_t ws_partials;         // bytes of the partial sums
  size_t ws_bytes;            // counters + partials (+ n * M * K * 2 of gathered x)
};

// Layout of one launch over n layers that share K on a device with
// `sm_count` SMs; false if this kernel cannot take them.
bool make_plan(const exq_weight* w, int n, int M, int sm_count, Plan& p) {
  if (M < 1 || M > 16 || n < 1 || n > kMaxLayers) return false;
  p.S = w[0].K / 32;
  if (p.S > 0xFFFF) return false;  // segment indices travel in 16 bits
  p.n_tiles = 0;
  p.gather = false;
  for (int i = 0; i < n; ++i) {
    p.tile0[i] = p.n_tiles;
    p.n_tiles += (w[i].N + kTN - 1) / kTN;
    p.gather = p.gather || w[i].perm != nullptr;
  }
  p.tile0[n] = p.n_tiles;
  if (p.n_tiles * kColGroups * 4 > kCounterBytes) return false;
  const long long total = static_cast<long long>(p.n_tiles) * p.S;
  if (total >= (1ll << 31)) return false;
  p.total = static_cast<int>(total);
  const size_t table = w[0].format != EXQ_FMT_GPTQ4 ? align_up(static_cast<size_t>(n) * (p.S + 1) * 4, 16) : 0;
  const size_t fixed = 512 + table + 1024;  // barriers and descriptors, the segment tables, alignment slack
  // EXL2 stages of 40 rows where two such slots fit half an SM;
  // EXQ_GEMV_ROWS=32 keeps them at 32 (a test hook: both heights are tested)
  const char* rows_env = std::getenv("EXQ_GEMV_ROWS");
  const bool long_fits = w[0].format != EXQ_FMT_GPTQ4 && M <= 8 &&
                         2 * static_cast<size_t>(slot_bytes_for(M, kRowsLong)) + fixed <= static_cast<size_t>(kSmemHalf);
  p.rows = long_fits && !(rows_env && std::atoi(rows_env) == kRowsShort) ? kRowsLong : kRowsShort;
  p.slot_bytes = slot_bytes_for(M, p.rows);
  // one set per CTA and two CTAs per SM where a ring of two slots fits half
  // the shared memory (M <= 8): a CTA of the next call can then start on an
  // SM while the other CTA there still works on this one
  p.sets = sets_of(M <= 8 ? 1 : 2);
  p.per_sm = p.sets == 1 && 2 * static_cast<size_t>(p.slot_bytes) + fixed <= static_cast<size_t>(kSmemHalf) ? 2 : 1;
  const long long budget = p.per_sm == 2 ? kSmemHalf : kSmemPerCta;
  int G = p.per_sm * sm_count;
  if (const char* env = std::getenv("EXQ_GEMV_CTAS")) {  // CTA-count override for tests of the split
    const int v = std::atoi(env);
    if (v > 0) G = v;
  }
  p.G = std::max(1, std::min(G, p.total));
  const long long room = budget - static_cast<long long>(fixed);
  p.stages = static_cast<int>(std::min<long long>(kMaxStages, room / p.slot_bytes));
  if (p.stages < 2) return false;
  p.off_bar = p.stages * p.slot_bytes;
  p.smem = static_cast<size_t>(p.off_bar) + fixed;
  // a tile of S units meets at most (S - 1) / s + 2 shares of at least s
  // units; each leaves one partial per consumer set
  const int min_share = std::max(1, p.total / p.G);
  p.max_pieces = p.sets * std::min(p.G, (p.S - 1) / min_share + 2);
  p.ws_partials = align_up(static_cast<size_t>(p.n_tiles) * p.max_pieces * M * kTP * 4, 256);
  p.ws_bytes = kCounterBytes + p.ws_partials +
               (p.gather ? align_up(static_cast<size_t>(n) * M * w[0].K * 2, 256) : 0);
  return true;
}

std::mutex g_attr_mutex;
bool g_attr_done[64][24];

}  // namespace

size_t gemv_workspace_bytes(const exq_weight* w, int n, int M) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  Plan plan{};
  if (!make_plan(w, n, M, device_info(dev).sm_count, plan)) return 0;
  return plan.ws_bytes;
}

exq_status launch_gemv(const exq_weight* w, int n, const uint16_t* x, int M, uint16_t* const* y, void* workspace,
                       size_t ws_bytes, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EXQ_ERR_CUDA;
  const DeviceInfo& di = device_info(dev);
  if (di.sm_count <= 0 || dev >= 64) return EXQ_ERR_CUDA;

  Plan plan{};
  if (!make_plan(w, n, M, di.sm_count, plan)) return EXQ_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < plan.ws_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return EXQ_ERR_INVALID_ARG;
  const exq_weight& w0 = w[0];

  const bool long_rows = plan.rows == kRowsLong;
  KernelFn fn = pick_kernel(w0.format, M, plan.gather, long_rows);
  {
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    bool& done = g_attr_done[dev][variant_index(w0.format, M, plan.gather, long_rows)];
    if (!done) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemPerCta) != cudaSuccess ||
          cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
        return EXQ_ERR_CUDA;
      done = true;
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

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // act-order: gather x into each layer's stored-row order once, into the workspace
  const uint16_t* xs_src = x;
  if (plan.gather) {
    uint16_t* xp = reinterpret_cast<uint16_t*>(ws + kCounterBytes + plan.ws_partials);
    GatherArgs ga{};
    for (int i = 0; i < n; ++i) {
      ga.perm[i] = w[i].perm;
      ga.seg_off[i] = w[i].seg_word_off;
    }
    const int threads = M * w0.K;  // per layer
    cudaLaunchConfig_t gcfg{};
    gcfg.gridDim = dim3((threads + 255) / 256, n, 1);
    gcfg.blockDim = dim3(256, 1, 1);
    gcfg.stream = stream;
    gcfg.attrs = attrs;
    gcfg.numAttrs = na;
    if (cudaLaunchKernelEx(&gcfg, gather_x_kernel, x, ga, M, w0.K, xp, w0.K / 32) != cudaSuccess) {
      cudaGetLastError();
      return EXQ_ERR_CUDA;
    }
    xs_src = xp;
  }

  GemvMaps maps;
  std::memset(&maps, 0, sizeof maps);
  GemvArgs args{};
  const int scale_rows = w0.format == EXQ_FMT_GPTQ4 ? w0.n_groups : w0.K / 32;
  for (int i = 0; i < kMaxLayers; ++i) {
    GemvLayer& l = args.L[i];
    if (i >= n) {
      l.tile0 = INT_MAX;
      continue;
    }
    // A tile's 992-byte word row starts on a 32-byte boundary, rarely on a
    // 256-byte one: with 256-byte L2 promotion each row pulled about 1216
    // bytes, and the edges again for the neighbouring tile (another CTA,
    // another time). 64-byte promotion cut the DRAM reads of a 70B gate+up
    // call from 1.146 to 1.091 times the packed bytes.
    if (!encode_2d(&maps.w[i], CU_TENSOR_MAP_DATA_TYPE_UINT32, w[i].qweight, w[i].N, w[i].n_word_rows,
                   static_cast<uint64_t>(w[i].N) * 4, kTN, plan.rows, CU_TENSOR_MAP_L2_PROMOTION_L2_64B))
      return EXQ_ERR_CUDA;
    // fp16 scale rows (two-level scales come without a tensor map)
    if (w[i].scales && !encode_2d(&maps.s[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, w[i].scales, w[i].N, scale_rows,
                                  static_cast<uint64_t>(w[i].N) * 2, kTN, kScaleRows,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_64B))
      return EXQ_ERR_CUDA;
    l.seg_off = w[i].seg_word_off;
    l.qzeros = w[i].qzeros;
    l.q_scale = w[i].q_scale;
    l.q_scale_max = w[i].q_scale_max;
    l.y = y[i];
    l.N = w[i].N;
    l.n_word_rows = w[i].n_word_rows;
    l.tile0 = plan.tile0[i];
    l.x_row = plan.gather ? i * M : 0;
  }
  if (!encode_2d(&maps.x, CU_TENSOR_MAP_DATA_TYPE_UINT16, xs_src, w0.K, static_cast<uint64_t>(plan.gather ? n : 1) * M,
                 static_cast<uint64_t>(w0.K) * 2, kXBox, M))
    return EXQ_ERR_CUDA;

  args.counters = reinterpret_cast<uint32_t*>(ws);
  args.partials = reinterpret_cast<float*>(ws + kCounterBytes);
  args.K = w0.K;
  args.M = M;
  args.S = plan.S;
  args.gs_seg = w0.format == EXQ_FMT_GPTQ4 ? w0.group_size / 32 : 1;
  args.G = w0.format == EXQ_FMT_GPTQ4 ? w0.n_groups : plan.S;
  args.n_tiles = plan.n_tiles;
  args.total = plan.total;
  args.max_pieces = plan.max_pieces;
  args.stages = plan.stages;
  args.slot_bytes = plan.slot_bytes;
  args.off_bar = plan.off_bar;
  const int starve = testing_starve_rounds();
  args.wait_limit = starve > 0 ? starve : kWaitLimit;
  args.sleep_limit = starve > 0 ? starve : kSleepLimit;
  args.starve = starve > 0 ? 1 : 0;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(plan.G, 1, 1);
  cfg.blockDim = dim3((plan.sets * kColGroups + 1) * 32, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, fn, maps, args) != cudaSuccess) {
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
