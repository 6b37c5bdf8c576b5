/*
 * exq.h -- C ABI of libexq, a dequantize-fused quantized matmul for sm_103a.
 *
 *   y[M, N] = x[M, K] . dequant(Wq)[K, N]      fp16 in, fp32 accumulate, fp16 out
 *
 * Three weight formats, as described by the ExLlamaV2 pages:
 *
 *  GPTQ 4-bit: group-wise codes q in 0..15, one fp16 scale s and one 4-bit
 *    zero z per (group, output column), w = (q - z) * s. Optional act-order:
 *    g_idx[k] assigns each input row k to a group; rows are stored sorted by
 *    group and a permutation maps stored rows back to input features.
 *    (ExLlamaV2 blog post "ExLlamaV2: The fastest inference engine for
 *    quantized Llama/HF models", section "How the Fused CUDA Kernel Works";
 *    ExLlamaV2 README, "Performance" table, act-order column.)
 *
 *  EXL2: rows are cut into 32-row segments, each packed at its own width
 *    b in {2,3,4,5,6,8}; symmetric codes, w = (q - 2^(b-1)) * s with one fp16
 *    scale per (segment, output column); a row permutation maps stored rows
 *    to input features. (ExLlamaV2 README, section "EXL2 quantization";
 *    blog post, "Step 3: Quantization Application".)
 *
 *  EXL2 with two-level scales: as EXL2, but the scale of (segment, column)
 *    is a 4-bit code c times the column's fp16 maximum m (the q_scale and
 *    q_scale_max tensors of the blog post's "Step 3: Quantization
 *    Application", multiplied together in "How the Fused CUDA Kernel
 *    Works"). The pages leave the code -> fraction map open; here code c is
 *    the fraction (c + 1) / 16, so c = 15 is the maximum, and the segment's
 *    fp16 scale is s = fp16_round_to_nearest_even(((c + 1) / 16) * m), then
 *    w = (q - 2^(b-1)) * s as for EXL2. Scale storage drops from 16 to 4 bits
 *    per (segment, column).
 *
 * Packed layouts (fixed by this library; the pages leave them open):
 *  - qweight is uint32 [n_word_rows, N], N contiguous (row-major), packing
 *    runs along K, least-significant bits first.
 *  - GPTQ: stored row j = 8r + i is nibble i (bits 4i..4i+3) of qweight[r][n].
 *    qzeros is uint32 [G, N/8]: zero of column n = 8c + i is nibble i of
 *    qzeros[g][c]. scales fp16 [G, N]. Group of stored row j is j / group_size.
 *  - EXL2: segment s occupies word rows [seg_word_off[s], seg_word_off[s+1]);
 *    its width is b = seg_word_off[s+1] - seg_word_off[s]. For column n the
 *    segment's 32 codes form a 32*b-bit stream, code i at stream bits
 *    [i*b, i*b+b), stream bit p is bit (p mod 32) of word row
 *    seg_word_off[s] + p/32. scales fp16 [S, N].
 *  - EXL2 two-level: q_scale is uint32 [S, N/8], the code of column
 *    n = 8k + i is nibble i of q_scale[s][k]; q_scale_max fp16 [N].
 *  - perm int32 [K] (optional): perm[j] = input feature (row of x's K axis
 *    and of the dequantized W) held by stored row j.
 *  - Dequantized weight: w = fp16_round_to_nearest_even((q - z) * s), computed
 *    with exactly one rounding.
 *
 * Conventions for every call below:
 *  - Device pointers are BORROWED: the caller allocates, owns and frees them.
 *    The library never allocates device or host memory and keeps no state
 *    between calls except one device-side error word.
 *  - Device calls are asynchronous on `stream` (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream) and never synchronise.
 *  - Argument checks run on the host before any launch; a failed check
 *    returns EXQ_ERR_INVALID_ARG or EXQ_ERR_UNSUPPORTED and launches nothing.
 *    A failed launch returns EXQ_ERR_CUDA.
 *  - Kernels that wait on on-chip barriers give up after a bounded time,
 *    record EXQ_ERR_TIMEOUT in the device error word and return; read it with
 *    exq_get_last_device_error().
 *  - Per-device set-up (kernel attributes, exq_gemm_noalloc's scratch
 *    address) is done on the first call on a device and kept; after
 *    cudaDeviceReset the process must not use the library on that device.
 *  - Device pointers must be 16-byte aligned; N % 8 == 0; GPTQ needs
 *    K % group_size == 0 and group_size % 32 == 0; EXL2 needs K % 32 == 0.
 *  - fp16 values travel as their uint16 bit patterns.
 */
#ifndef EXQ_H
#define EXQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EXQ_OK = 0,
  EXQ_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or layout        */
  EXQ_ERR_UNSUPPORTED = 2, /* valid, but outside what this build handles    */
  EXQ_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed          */
  EXQ_ERR_TIMEOUT = 4      /* a device-side wait gave up (from the device)  */
} exq_status;

typedef enum { EXQ_FMT_GPTQ4 = 1, EXQ_FMT_EXL2 = 2, EXQ_FMT_EXL2_QSCALE = 3 } exq_format;

/* Plain descriptor of one packed linear layer. Every pointer is a borrowed
 * DEVICE pointer. */
typedef struct {
  int32_t format;      /* exq_format                                          */
  int32_t K;           /* input features (rows of W)                          */
  int32_t N;           /* output features (columns of W)                      */
  int32_t group_size;  /* GPTQ: rows per group (multiple of 32); EXL2: 32     */
  int32_t n_groups;    /* GPTQ: G = K / group_size; EXL2: S = K / 32           */
  int32_t n_word_rows; /* rows of qweight: GPTQ K / 8; EXL2 sum of widths     */
  const uint32_t* qweight;      /* [n_word_rows, N]                           */
  const uint16_t* scales;       /* fp16 [n_groups, N]; EXL2 two-level: NULL   */
  const uint32_t* qzeros;       /* GPTQ: [G, N/8]; EXL2: NULL                 */
  const int32_t* perm;          /* [K] stored row -> input feature, or NULL   */
  const uint32_t* seg_word_off; /* EXL2 (both): [S + 1] word-row prefix sums; GPTQ: NULL */
  const uint32_t* q_scale;      /* EXL2 two-level: [S, N/8] 4-bit codes; else NULL */
  const uint16_t* q_scale_max;  /* EXL2 two-level: fp16 [N] column maxima; else NULL */
} exq_weight;

/* ---------------------------------------------------------------- packers */

/* exq_pack_gptq -- host-only, synchronous, no CUDA.
 * Packs a GPTQ layer (ExLlamaV2 blog post, "How the Fused CUDA Kernel Works":
 * eight 4-bit codes per uint32, least-significant nibble first).
 *   q      [K, N] uint8 codes 0..15, rows in input-feature order (host)
 *   z      [G, N] uint8 zero points 0..15 (host), G = K / group_size
 *   g_idx  [K] group of each input row, or NULL for k / group_size (host).
 *          Every group must hold exactly group_size rows.
 *   qweight_out [K/8, N], qzeros_out [G, N/8], perm_out [K] (host, caller-
 *          allocated). Rows are stored sorted stably by (g_idx[k], k) and
 *          perm_out[j] is the input row of stored row j. The fp16 scales
 *          [G, N] need no packing and are used as they are.
 * Returns EXQ_ERR_INVALID_ARG for NULL buffers, K % group_size, N % 8,
 * K % 8, a code or zero above 15, or a malformed g_idx; outputs are then
 * unspecified. */
exq_status exq_pack_gptq(const uint8_t* q, const uint8_t* z, const int32_t* g_idx,
                         int32_t K, int32_t N, int32_t group_size,
                         uint32_t* qweight_out, uint32_t* qzeros_out, int32_t* perm_out);

/* exq_pack_exl2 -- host-only, synchronous, no CUDA.
 * Packs an EXL2 layer (ExLlamaV2 README, "EXL2 quantization"; blog post,
 * "Step 3: Quantization Application") into the segment bit streams above.
 *   q      [K, N] uint8 codes in STORED row order, code < 2^bits[j/32] (host)
 *   bits   [S] widths in {2,3,4,5,6,8}, S = K / 32 (host)
 *   qweight_out [sum(bits), N] (host, caller-allocated; size from
 *          exq_exl2_word_rows), seg_word_off_out [S + 1] (host).
 * The fp16 scales [S, N] and the permutation need no packing.
 * Returns EXQ_ERR_INVALID_ARG for NULL buffers, K % 32, N % 8, a width
 * outside the set or a code that does not fit its width. */
exq_status exq_pack_exl2(const uint8_t* q, const uint8_t* bits, int32_t K, int32_t N,
                         uint32_t* qweight_out, uint32_t* seg_word_off_out);

/* exq_pack_exl2_qscale -- host-only, synchronous, no CUDA.
 * Packs the 4-bit scale codes of an EXL2 two-level layer.
 *   codes  [S, N] uint8 codes 0..15, one per (segment, output column) (host)
 *   q_scale_out [S, N/8] uint32 (host, caller-allocated): nibble i of word k
 *          is the code of column 8k + i.
 * Returns EXQ_ERR_INVALID_ARG for NULL buffers, S <= 0, N <= 0, N % 8 or a
 * code above 15. */
exq_status exq_pack_exl2_qscale(const uint8_t* codes, int32_t S, int32_t N, uint32_t* q_scale_out);

/* Number of qweight rows an EXL2 layer needs: sum of bits[0..n_segments).
 * Returns -1 if bits is NULL, n_segments <= 0 or a width is outside the set. */
int64_t exq_exl2_word_rows(const uint8_t* bits, int32_t n_segments);

/* exq_exl2_seg_word_off -- host-only, synchronous, no CUDA.
 * The segment table of an EXL2 layer (the row remapping of the ExLlamaV2
 * README, "EXL2 quantization", stores each segment's words after the previous
 * one's): seg_word_off_out[s] = bits[0] + ... + bits[s-1] for s = 0..S, so
 * segment s occupies word rows [seg_word_off_out[s], seg_word_off_out[s+1]).
 *   bits  [S] widths in {2,3,4,5,6,8} (host)
 *   seg_word_off_out [S + 1] uint32 (host, caller-allocated)
 * exq_pack_exl2 writes the same table; this call serves callers that lay
 * out the words themselves (exq_quantize_exl2 takes the table as input).
 * Returns EXQ_ERR_INVALID_ARG for NULL buffers, S <= 0 or a width outside
 * the set. */
exq_status exq_exl2_seg_word_off(const uint8_t* bits, int32_t n_segments, uint32_t* seg_word_off_out);

/* ---------------------------------------------------------------- device ops */

/* exq_dequant -- W_out[perm[j]][n] = w(j, n) for every stored row j, i.e. the
 * dense fp16 weight [K, N] in input-feature order, bit-exact to the
 * definition above (the "dequantize first" path the ExLlamaV2 blog post,
 * "Finding 2", contrasts with the fused kernel).
 *   w      descriptor with device pointers (host struct, read during the call)
 *   W_out  device fp16 [K, N], caller-allocated, fully overwritten */
exq_status exq_dequant(const exq_weight* w, uint16_t* W_out, void* stream);

/* Bytes of device workspace exq_gemv needs for this layer and M on the
 * current device (it depends on the SM count); 0 for an invalid layer or M
 * outside 1..16. */
size_t exq_gemv_workspace_size(const exq_weight* w, int32_t M);

/* exq_gemv -- decode-sized fused matmul, 1 <= M <= 16 (ExLlamaV2 blog post,
 * "How the Fused CUDA Kernel Works": the packed weights are read once,
 * dequantized in registers and multiplied into fp32 sums).
 *   x  device fp16 [M, K] row-major, input-feature order
 *   y  device fp16 [M, N] row-major, fully overwritten
 *   workspace  device buffer of at least exq_gemv_workspace_size() bytes,
 *              256-byte aligned. Its first 64 KB hold per-tile counters of
 *              the split over SMs: ZERO-FILL them before the first use; every
 *              call that completes leaves them zero again, so one workspace
 *              serves any sequence of calls (any layer, any M) ordered on one
 *              stream. The rest is scratch (partial sums and, for a permuted
 *              layer, x gathered into stored-row order). Calls that may
 *              overlap on the GPU need separate workspaces. A call that ends
 *              in EXQ_ERR_TIMEOUT (exq_get_last_device_error) may leave
 *              counters non-zero: zero-fill the first 64 KB again before the
 *              workspace serves another call.
 * Deterministic: the same inputs give the same bits.
 * Returns EXQ_ERR_UNSUPPORTED for M > 16 (use exq_gemm) and
 * EXQ_ERR_INVALID_ARG for a missing, short or misaligned workspace. */
exq_status exq_gemv(const exq_weight* w, const uint16_t* x, int32_t M, uint16_t* y,
                    void* workspace, size_t ws_bytes, void* stream);

/* Most layers one exq_gemv_multi call takes. */
#define EXQ_GEMV_MAX_LAYERS 4

/* Bytes of device workspace exq_gemv_multi needs for these n layers and M on
 * the current device; 0 for an invalid group (see exq_gemv_multi) or M
 * outside 1..16. exq_gemv_workspace_size(w, M) equals this with n = 1. */
size_t exq_gemv_multi_workspace_size(const exq_weight* w, int32_t n, int32_t M);

/* exq_gemv_multi -- several decode matmuls that read the same activations,
 * y_i = x . dequant(Wq_i) for i < n, in ONE launch: the q, k and v
 * projections of an attention block, or the gate and up projections of an
 * MLP. The architecture figure of the ExLlamaV2 blog post (section "The
 * Solution", CUDA kernel layer) has the QKV projection as one kernel; here
 * the layers stay separate tensors and only their work is pooled, so the SMs
 * split the layers' combined weight stream evenly and the call pays one
 * start-up and one tail instead of n.
 *   w  host array of n descriptors (device pointers), 1 <= n <=
 *      EXQ_GEMV_MAX_LAYERS, read during the call. All of one format, with
 *      the same K and (GPTQ) the same group_size; N, the permutation (or
 *      none) and every pointer may differ.
 *   x  device fp16 [M, K], input-feature order, shared by every layer
 *   y  host array of n device pointers, y[i] fp16 [M, w[i].N], fully
 *      overwritten; the outputs must not overlap one another or x
 *   workspace  as for exq_gemv, at least exq_gemv_multi_workspace_size()
 *      bytes; the same zero-filled counters serve exq_gemv and
 *      exq_gemv_multi calls in any order on one stream.
 * Each y[i] is what exq_gemv gives for layer i up to the order of the fp32
 * additions (the split over SMs differs), and the call is deterministic.
 * The columns of all layers together may use at most 2048 tiles of 248
 * columns (sum of N up to 507,904), else EXQ_ERR_UNSUPPORTED.
 * Returns EXQ_ERR_INVALID_ARG for a bad n, a layer that fails the checks of
 * exq_gemv, mixed formats, K or group sizes, or a bad output pointer. */
exq_status exq_gemv_multi(const exq_weight* w, int32_t n, const uint16_t* x, int32_t M,
                          uint16_t* const* y, void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device workspace exq_gemm needs for this layer and M (0 if none).
 * Two parts, both scratch: for a permuted layer, M * K * 2 bytes (rounded up
 * to 256) of activations gathered into stored-row order; and, when the grid
 * of 128-column x 256-token tiles is too small to fill the GPU (fewer tiles
 * than half the SMs), split * M * N * 4 bytes of fp32 partial sums of a K
 * split (split <= 8, each split at least 512 rows of K). The size is the
 * largest any device (up to 256 SMs) would use, so it does not depend on the
 * current device. */
size_t exq_gemm_workspace_size(const exq_weight* w, int32_t M);

/* exq_gemm -- prefill-sized fused matmul for any M >= 1 (tuned for M >= 128).
 * The ExLlamaV2 blog post ("How the Fused CUDA Kernel Works", the paragraph
 * after the conceptual kernel) says the real kernel handles several widths
 * and uses tensor cores while keeping the same fused shape: packed weights
 * are loaded, dequantized on the fly and multiplied, with no dense weight
 * written to memory. Here that is
 * computed as y^T = W^T x^T on the tcgen05 tensor cores, the packed weights
 * dequantized to fp16 straight into tensor memory as the A operand, x read
 * by TMA as the B operand, fp32 accumulation in tensor memory.
 *   x  device fp16 [M, K], y device fp16 [M, N] (fully overwritten)
 *   workspace  device buffer of at least exq_gemm_workspace_size() bytes
 *              (may be NULL when that size is 0); contents are scratch.
 *              Calls that may overlap on the GPU need separate workspaces.
 * With a K split a second kernel adds the splits' partial sums in split
 * order: the same inputs give the same bits on the same device.
 * Requires K % 64 == 0 and N % 128 == 0 in addition to the rules above,
 * else EXQ_ERR_UNSUPPORTED; a missing, short or misaligned workspace is
 * EXQ_ERR_INVALID_ARG. */
exq_status exq_gemm(const exq_weight* w, const uint16_t* x, int32_t M, uint16_t* y,
                    void* workspace, size_t ws_bytes, void* stream);

/* Most layers one exq_gemm_multi call takes. */
#define EXQ_GEMM_MAX_LAYERS 4

/* Bytes of device workspace exq_gemm_multi needs for these n layers and M:
 * n * M * K * 2 bytes (rounded up to 256) of activations gathered into each
 * layer's stored-row order when any of the layers has a permutation, plus
 * the fp32 partial sums of the largest K split that any one of the layers
 * would take alone (as in exq_gemm_workspace_size). 0 when neither applies,
 * and for an invalid group (see exq_gemm_multi). */
size_t exq_gemm_multi_workspace_size(const exq_weight* w, int32_t n, int32_t M);

/* exq_gemm_multi -- several prefill matmuls that read the same activations,
 * y_i = x . dequant(Wq_i) for i < n, in ONE launch: the q, k and v
 * projections of an attention block, or the gate and up projections of an
 * MLP (the architecture figure of the ExLlamaV2 blog post, section "The
 * Solution", has the QKV projection as one kernel). The layers stay separate
 * tensors; their 128-column tiles are pooled in one grid, so a small layer
 * (the 1024-column k and v of a grouped-query model) shares the GPU with the
 * large one instead of running alone on a few SMs.
 *   w  host array of n descriptors, 1 <= n <= EXQ_GEMM_MAX_LAYERS, all of one
 *      format with the same K and (GPTQ) group size; each N % 128 == 0 and
 *      K % 64 == 0, else EXQ_ERR_UNSUPPORTED. Permutations may differ.
 *   x  device fp16 [M, K], input-feature order, shared by every layer
 *   y  host array of n device pointers, y[i] fp16 [M, w[i].N], fully
 *      overwritten; they must not overlap one another or x
 *   workspace  at least exq_gemm_multi_workspace_size() bytes (may be NULL
 *      when that is 0); scratch; calls that may overlap on the GPU need
 *      separate workspaces.
 * The call picks, from the shapes and the device's SM count, one launch over
 * the pooled tiles or one launch per layer, whichever fills the SMs in fewer
 * waves (one launch per layer splits K for a small layer as exq_gemm does);
 * x is gathered once either way. Each y[i] has the bits of exq_gemm on
 * layer i, or of its unsplit form when exq_gemm would split K and the group
 * is pooled (they differ at most in the last bit). Deterministic for given
 * shapes and device. Returns EXQ_ERR_INVALID_ARG for a bad n, mixed formats,
 * K or group sizes, a bad pointer or a short workspace. */
exq_status exq_gemm_multi(const exq_weight* w, int32_t n, const uint16_t* x, int32_t M,
                          uint16_t* const* y, void* workspace, size_t ws_bytes, void* stream);

/* exq_gemm_noalloc -- exq_gemm for callers that cannot allocate device memory.
 * The ExLlamaV2 pages have no counterpart; this is a deployment variant.
 * Some callers cannot hand the library a workspace: inference-runtime plugins
 * whose enqueue path must not allocate because the host framework plans all
 * device memory up front, and serving loops that cannot afford cudaMalloc's
 * implicit device-wide synchronisation. For them this call takes the gathered
 * activations of an act-order layer from a scratch array that the library
 * reserves statically: EXQ_NOALLOC_SCRATCH_BYTES on every GPU that loads
 * libexq, kept until the process exits. Layers without a permutation need no
 * scratch at all.
 *   Same arguments and results as exq_gemm without the workspace, except
 *   that it never splits K (the partial sums would need more scratch), so
 *   grids of few tiles run slower and may round differently in the last bit.
 *   Returns EXQ_ERR_UNSUPPORTED (and launches nothing) if the layer has a
 *   permutation and M * K * 2 > EXQ_NOALLOC_SCRATCH_BYTES.
 *   The array is part of the library's GEMM module, so the CUDA driver
 *   commits it when that module loads on a device: with lazy module loading
 *   (CUDA's default) that is during the first exq_gemm or exq_gemm_noalloc
 *   call there. The first exq_gemm_noalloc call on a device, with or without
 *   a permutation, also looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current). So make one call on
 *   each device before any stream capture. The call itself allocates
 *   nothing, then or later.
 *   Every call on a device shares the one array, which keeps the previous
 *   call's contents (the array is fully rewritten before it is read, so
 *   nothing needs clearing). Calls whose kernels overlap on the GPU (other
 *   streams, other host threads) race on it: order them on one stream. */
#define EXQ_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
exq_status exq_gemm_noalloc(const exq_weight* w, const uint16_t* x, int32_t M, uint16_t* y, void* stream);

/* ---------------------------------------------------------------- quantized KV cache */

/* Quantized KV cache codec, Q4 / Q6 / Q8 (ExLlamaV2 blog post: comparison
 * table and "Step 2: Use the right cache mode for your context length" name
 * the Q4 / Q6 / Q8 cache; "Production Considerations" costs it at half a byte
 * and one byte per element for Q4 / Q8). The pages do not describe the codec;
 * this one quantises groups of D values (one token's one head of K or V),
 * symmetric, qmax = 2^(bits-1) - 1:
 *   s = fp16_RNE(fp32_RNE(amax / qmax)),
 *   q = clamp(rint(fp32_RNE(x / s)), -qmax - 1, qmax)   (q = 0 where s = 0),
 *   stored code u = q + 2^(bits-1); code i of a group at bits
 *   [i*bits, i*bits + bits) of the group's little-endian uint32 stream;
 *   read back as fp16_RNE((u - 2^(bits-1)) * s).
 * rint rounds half to even. Inputs must be finite.
 *   x       device fp16 [n_groups, D]
 *   codes   device uint32 [n_groups, D * bits / 32]
 *   scales  device fp16 [n_groups]
 * D must be 64, 128 or 256 and bits 4, 6 or 8, else EXQ_ERR_UNSUPPORTED;
 * n_groups < 0, a NULL or misaligned pointer (16 bytes) is EXQ_ERR_INVALID_ARG;
 * n_groups = 0 launches nothing and returns EXQ_OK (the pointers are then not
 * looked at and may be NULL). Outputs are fully overwritten; the same
 * inputs give the same bits. */
exq_status exq_kv_quantize(const uint16_t* x, int64_t n_groups, int32_t D, int32_t bits, uint32_t* codes,
                           uint16_t* scales, void* stream);

/* exq_kv_dequantize -- the inverse read: x_out fp16 [n_groups, D] from codes
 * and scales as written by exq_kv_quantize (same argument rules). */
exq_status exq_kv_dequantize(const uint32_t* codes, const uint16_t* scales, int64_t n_groups, int32_t D,
                             int32_t bits, uint16_t* x_out, void* stream);

/* ---------------------------------------------------------------- EXL2 conversion */

/* Converting an fp16 weight to EXL2 without calibration data (ExLlamaV2 blog
 * post, "How the EXL2 Quantization Pipeline Works Under the Hood": Step 1
 * measures each layer at every width, Step 2 solves for a width per group at a
 * target bpw, Step 3 quantises). The measurement on calibration text is out of
 * reach here; it is stood in for by the weight-space squared error of a
 * round-to-nearest quantisation. The quantiser is symmetric per (32-row
 * segment, column), qmax = 2^(b-1) - 1:
 *   s = fp16_RNE(fp32_RNE(amax / qmax)),
 *   q = clamp(rint(fp32_RNE(w / s)), -qmax - 1, qmax)   (q = 0 where s = 0),
 *   stored code u = q + 2^(b-1), i.e. the EXL2 dequantisation gives back
 *   fp16_RNE(q * s). */

/* exq_quantize_exl2 -- device, asynchronous.
 *   W            device fp16 [K, N], input-feature order
 *   perm         device int32 [K] (stored row j holds input row perm[j]) or NULL
 *   seg_word_off device uint32 [K/32 + 1]: the widths as prefix sums (see the
 *                EXL2 layout; exq_pack_exl2 returns them, or build them from
 *                the solve's widths)
 *   n_word_rows  seg_word_off[K/32] (rows of qweight_out)
 *   qweight_out  device uint32 [n_word_rows, N], scales_out device fp16 [K/32, N]
 * The result is an EXL2 layer (with perm) for exq_gemv / exq_gemm / exq_dequant.
 * A width outside the set, or offsets past n_word_rows, leave that segment
 * unwritten and set EXQ_ERR_INVALID_ARG in the device error word; so do
 * permutation entries outside [0, K) (read as 0). */
exq_status exq_quantize_exl2(const uint16_t* W, const int32_t* perm, int32_t K, int32_t N,
                             const uint32_t* seg_word_off, int32_t n_word_rows, uint32_t* qweight_out,
                             uint16_t* scales_out, void* stream);

/* Bytes of device workspace exq_measure_exl2 needs (0 for bad K, N). */
size_t exq_measure_exl2_workspace_size(int32_t K, int32_t N);

/* exq_measure_exl2 -- device, asynchronous: err_out fp32 [K/32, 6], the sum
 * over a segment's 32 x N weights of (w - w_hat)^2 at widths 2, 3, 4, 5, 6, 8
 * (w_hat the fp16 dequantisation of the RTN codes above). fp32 sums in a
 * fixed order: deterministic. Same W / perm rules as exq_quantize_exl2. */
exq_status exq_measure_exl2(const uint16_t* W, const int32_t* perm, int32_t K, int32_t N, float* err_out,
                            void* workspace, size_t ws_bytes, void* stream);

/* exq_solve_exl2_bits -- host, synchronous: widths for a budget of code bits.
 *   err     host double [S, 6], the error table (exq_measure_exl2's, or any)
 *   budget  total code bits per column, sum of the widths (e.g. bpw * S)
 *   bits_out host uint8 [S]
 * Every segment starts at 2 bits; while some step to the next width (2, 3,
 * 4, 5, 6, 8) fits the budget, the step with the largest
 * (err[b] - err[b_next]) / (b_next - b) is taken, the lowest segment on
 * ties (the increase loop of the blog post's Step 2 greedy, started from the
 * smallest width). Returns EXQ_ERR_INVALID_ARG for NULL buffers, S <= 0 or a
 * budget below 2 * S. */
exq_status exq_solve_exl2_bits(const double* err, int32_t S, int64_t budget, uint8_t* bits_out);

/* ---------------------------------------------------------------- status */

/* Static, NUL-terminated description of a status code. */
const char* exq_status_string(exq_status s);

/* Synchronises `stream`, then returns and clears the device error word of the
 * current device: EXQ_OK, EXQ_ERR_TIMEOUT (a kernel gave up waiting) or
 * EXQ_ERR_INVALID_ARG (a kernel met an EXL2 segment width outside the set or
 * past the end of qweight, or a permutation entry outside [0, K)).
 * Returns EXQ_ERR_CUDA if the synchronisation itself fails. */
exq_status exq_get_last_device_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EXQ_H */
