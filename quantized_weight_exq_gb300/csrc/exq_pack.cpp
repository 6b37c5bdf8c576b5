// Host-side packers for the two weight formats (CPU only, no CUDA).
//
// GPTQ: eight 4-bit codes per uint32 along K, least-significant nibble first,
// as in the unpack `(packed >> 4i) & 0xF` of the ExLlamaV2 blog post
// ("ExLlamaV2: The fastest inference engine for quantized Llama/HF models",
// section "How the Fused CUDA Kernel Works"); act-order rows are stored
// sorted by group with a permutation back to input features (ExLlamaV2
// README, "Performance", act-order column, and "EXL2 quantization": the row
// remapping trick).
//
// EXL2: 32-row segments at widths {2,3,4,5,6,8} (README, "EXL2
// quantization"); each segment-column is a 32*b-bit little-endian stream.
#include <queue>
#include <utility>
#include <vector>
#include <cstdint>
#include <cstring>
#include <vector>

#include "exq.h"

namespace {

bool valid_exl2_width(unsigned b) {
  return b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8;
}

}  // namespace

extern "C" exq_status exq_pack_gptq(const uint8_t* q, const uint8_t* z, const int32_t* g_idx,
                                    int32_t K, int32_t N, int32_t group_size,
                                    uint32_t* qweight_out, uint32_t* qzeros_out,
                                    int32_t* perm_out) {
  if (!q || !z || !qweight_out || !qzeros_out || !perm_out) return EXQ_ERR_INVALID_ARG;
  if (K <= 0 || N <= 0 || group_size <= 0) return EXQ_ERR_INVALID_ARG;
  if (K % 8 || N % 8 || group_size % 8 || K % group_size) return EXQ_ERR_INVALID_ARG;
  const int64_t G = K / group_size;

  // stored order: counting sort by group, ties by ascending input row
  std::vector<int64_t> fill(G, 0);
  for (int64_t k = 0; k < K; ++k) {
    const int64_t g = g_idx ? g_idx[k] : k / group_size;
    if (g < 0 || g >= G) return EXQ_ERR_INVALID_ARG;
    if (fill[g] == group_size) return EXQ_ERR_INVALID_ARG;
    perm_out[g * group_size + fill[g]++] = static_cast<int32_t>(k);
  }

  for (int64_t r = 0; r < K / 8; ++r) {
    uint32_t* dst = qweight_out + r * N;
    std::memset(dst, 0, sizeof(uint32_t) * N);
    for (int i = 0; i < 8; ++i) {
      const uint8_t* src = q + static_cast<int64_t>(perm_out[8 * r + i]) * N;
      for (int64_t n = 0; n < N; ++n) {
        if (src[n] > 15) return EXQ_ERR_INVALID_ARG;
        dst[n] |= static_cast<uint32_t>(src[n]) << (4 * i);
      }
    }
  }
  for (int64_t g = 0; g < G; ++g) {
    for (int64_t c = 0; c < N / 8; ++c) {
      uint32_t word = 0;
      for (int i = 0; i < 8; ++i) {
        const uint8_t v = z[g * N + 8 * c + i];
        if (v > 15) return EXQ_ERR_INVALID_ARG;
        word |= static_cast<uint32_t>(v) << (4 * i);
      }
      qzeros_out[g * (N / 8) + c] = word;
    }
  }
  return EXQ_OK;
}

extern "C" int64_t exq_exl2_word_rows(const uint8_t* bits, int32_t n_segments) {
  if (!bits || n_segments <= 0) return -1;
  int64_t total = 0;
  for (int32_t s = 0; s < n_segments; ++s) {
    if (!valid_exl2_width(bits[s])) return -1;
    total += bits[s];
  }
  return total;
}

// Segment word offsets of an EXL2 layer: the prefix sums of its widths.
extern "C" exq_status exq_exl2_seg_word_off(const uint8_t* bits, int32_t n_segments, uint32_t* seg_word_off_out) {
  if (!seg_word_off_out || exq_exl2_word_rows(bits, n_segments) < 0) return EXQ_ERR_INVALID_ARG;
  uint32_t off = 0;
  for (int32_t s = 0; s < n_segments; ++s) {
    seg_word_off_out[s] = off;
    off += bits[s];
  }
  seg_word_off_out[n_segments] = off;
  return EXQ_OK;
}

extern "C" exq_status exq_pack_exl2(const uint8_t* q, const uint8_t* bits, int32_t K, int32_t N,
                                    uint32_t* qweight_out, uint32_t* seg_word_off_out) {
  if (!q || !bits || !qweight_out || !seg_word_off_out) return EXQ_ERR_INVALID_ARG;
  if (K <= 0 || N <= 0 || K % 32 || N % 8) return EXQ_ERR_INVALID_ARG;
  const int32_t S = K / 32;
  if (exq_exl2_word_rows(bits, S) < 0) return EXQ_ERR_INVALID_ARG;

  uint32_t off = 0;
  for (int32_t s = 0; s < S; ++s) {
    seg_word_off_out[s] = off;
    const unsigned b = bits[s];
    const uint32_t limit = 1u << b;
    uint32_t* rows = qweight_out + static_cast<int64_t>(off) * N;
    for (int64_t n = 0; n < N; ++n) {
      // accumulate the column's stream in a 64-bit window, emit whole words
      uint64_t window = 0;
      unsigned have = 0, word = 0;
      for (int i = 0; i < 32; ++i) {
        const uint32_t v = q[(static_cast<int64_t>(s) * 32 + i) * N + n];
        if (v >= limit) return EXQ_ERR_INVALID_ARG;
        window |= static_cast<uint64_t>(v) << have;
        have += b;
        if (have >= 32) {
          rows[static_cast<int64_t>(word++) * N + n] = static_cast<uint32_t>(window);
          window >>= 32;
          have -= 32;
        }
      }
    }
    off += b;
  }
  seg_word_off_out[S] = off;
  return EXQ_OK;
}

// Two-level EXL2 scale codes: eight 4-bit codes per word along N, least
// significant nibble first (the layout of the GPTQ zero points).
extern "C" exq_status exq_pack_exl2_qscale(const uint8_t* codes, int32_t S, int32_t N, uint32_t* q_scale_out) {
  if (!codes || !q_scale_out || S <= 0 || N <= 0 || N % 8) return EXQ_ERR_INVALID_ARG;
  for (int64_t s = 0; s < S; ++s)
    for (int32_t k = 0; k < N / 8; ++k) {
      uint32_t word = 0;
      for (int i = 0; i < 8; ++i) {
        const uint8_t v = codes[s * N + 8 * k + i];
        if (v > 15) return EXQ_ERR_INVALID_ARG;
        word |= static_cast<uint32_t>(v) << (4 * i);
      }
      q_scale_out[s * (N / 8) + k] = word;
    }
  return EXQ_OK;
}

// Widths for a budget of code bits: from 2 bits everywhere, repeatedly the
// step with the largest error decrease per added bit that still fits, the
// lowest segment on ties. A step that does not fit never will (the room only
// shrinks), so it leaves the queue for good.
extern "C" exq_status exq_solve_exl2_bits(const double* err, int32_t S, int64_t budget, uint8_t* bits_out) {
  static const int kW[6] = {2, 3, 4, 5, 6, 8};
  if (!err || !bits_out || S <= 0 || budget < 2 * static_cast<int64_t>(S)) return EXQ_ERR_INVALID_ARG;
  std::vector<int> level(S, 0);
  // (gain, -segment): the largest gain first, then the lowest segment
  using Item = std::pair<double, int32_t>;
  std::priority_queue<Item> heap;
  auto push = [&](int32_t s) {
    const int lv = level[s];
    if (lv + 1 < 6) heap.push({(err[6 * static_cast<int64_t>(s) + lv] - err[6 * static_cast<int64_t>(s) + lv + 1]) /
                                   (kW[lv + 1] - kW[lv]),
                               -s});
  };
  for (int32_t s = 0; s < S; ++s) push(s);
  int64_t total = 2 * static_cast<int64_t>(S);
  while (!heap.empty()) {
    const Item top = heap.top();
    heap.pop();
    const int32_t s = -top.second;
    const int step = kW[level[s] + 1] - kW[level[s]];
    if (total + step > budget) continue;
    total += step;
    ++level[s];
    push(s);
  }
  for (int32_t s = 0; s < S; ++s) bits_out[s] = static_cast<uint8_t>(kW[level[s]]);
  return EXQ_OK;
}
