"""CPU oracle for the dequantize-fused quantized matmul y = x . dequant(Wq).

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it. It shares
no code with the CUDA library (no headers, helpers, tables or kernels); the
two meet only at the packed-buffer layout, which both sides implement
independently from the format definition below.

It is deliberately plain and slow: bits are packed and unpacked one at a time,
each weight is dequantised by its definition and rounded to fp16 by an
IEEE-754 round-to-nearest-even written out here, and the matmul is a float64
``numpy.matmul``. Every function is pinned by ``tests/test_oracle_pins.py``
against values and properties fixed independently of this file (hand-derived
fixtures, numpy's own float16 conversion, exact integer arithmetic, one-hot
inputs, permutation invariance, cross-format reduction, brute force).

Sources (the ExLlamaV2 pages):
* ExLlamaV2 blog post ("ExLlamaV2: The fastest inference engine for
  quantized Llama/HF models"), section "How the Fused CUDA Kernel Works":
  each 4-bit code is ``(packed >> 4i) & 0xF`` (least-significant nibble
  first), it is dequantised as ``(code - zero) * scale`` in float, products are
  summed in float and the output is stored as fp16.
* Same post, "How the EXL2 Quantization Pipeline Works Under the Hood",
  "Step 3: Quantization Application": an EXL2 tensor is packed
  variable-bit-width codes plus scales, per-group bit widths and a row
  permutation for act-order compatibility.
* ExLlamaV2 README (exllamav2_Rocm mirror), section "EXL2 quantization":
  2, 3, 4, 5, 6 and 8-bit codes may be mixed inside one linear layer, and the
  same row-remapping used for act-order GPTQ models carries the mix.

Readings where the pages are silent:
* Packed weights are [K/8, N] (GPTQ) or [sum(bits), N] (EXL2) uint32 words,
  N contiguous; packing runs along K, least-significant bits first.
* EXL2 segment = 32 consecutive stored rows at one bit width b. For each
  column the segment's 32 codes form a 32*b-bit stream, code i at stream bits
  [i*b, i*b+b); stream bit p lives in bit (p mod 32) of word
  ``seg_word_off[s] + p // 32``. Segments are stored in stored-row order.
* GPTQ zero points are stored as the zero itself (no +1 offset), 4 bits,
  packed 8 per uint32 along N. EXL2 is symmetric: zero = 2^(b-1).
* GPTQ scales are fp16 [G, N]; EXL2 scales are fp16 [S, N], one per
  (segment, column).
* EXL2 with two-level scales (the q_scale / q_scale_max pair of "Step 3:
  Quantization Application", multiplied together in "How the Fused CUDA
  Kernel Works"): a 4-bit code c per (segment, column), packed 8 per uint32
  along N (nibble i of word k = column 8k + i), and one fp16 maximum m per
  column. The pages do not say how a code maps to a fraction; the reading
  here is (c + 1) / 16, so c = 15 is the maximum. The pages multiply
  (w - 8) * scale * scale_max in float, where the product is exact (at most
  8 + 5 + 11 significant bits), so the segment's scale s = ((c + 1) / 16) * m
  is kept exact, never rounded to fp16 on its own, and the weight is
  w = fp16_RNE((q - z) * s): one rounding, as for fp16 scales.
* Dequantised weight w = fp16_RNE((q - z) * s): the product is exact in
  float32 and float64 (at most 8 + 11 significant bits), so there is exactly
  one rounding.
* Act-order: ``g_idx[k]`` is the group of original row k; rows are stored
  sorted stably by (g_idx[k], k); ``perm[j]`` is the original row of stored
  row j. Every group must hold exactly ``group_size`` rows.
* The output is y = x . W accumulated in float64 here; the device path rounds
  its fp32 accumulator to fp16 once.
* Quantized KV cache (Q4 / Q6 / Q8: the blog post's comparison table, "Step 2:
  Use the right cache mode for your context length" and the VRAM estimate of
  "Production Considerations", which give only the bytes per element). The
  codec is not described; the reading here: a group is the D values of one
  (token, head), symmetric with qmax = 2^(b-1) - 1,
  s = fp16_RNE(fp32_RNE(amax / qmax)), q = clamp(rint(fp32_RNE(x / s)),
  -qmax - 1, qmax) (q = 0 where s = 0), stored u = q + 2^(b-1) as a b-bit
  code, code i at bits [i*b, i*b+b) of the group's little-endian word
  stream, read back as fp16_RNE((u - 2^(b-1)) * s). The integer decisions are
  taken in IEEE fp32 (numpy float32 division and rint), as on the device.
* EXL2 conversion without calibration data (blog post, "How the EXL2
  Quantization Pipeline Works Under the Hood", Steps 1-3): the measurement
  pass runs the model on calibration text, which is out of reach here; it is
  stood in for by the weight-space squared error of a round-to-nearest
  quantisation of each 32-row segment at each width (same symmetric RTN
  arithmetic as the KV codec, one group = one segment of one column). The
  solve pass follows the printed greedy's increase loop (take the step with
  the largest error decrease per added bit while the budget allows), started
  from every segment at the smallest width: started at 4 bits, as printed,
  it would leave a 4.0 bpw target unmixed. Ties go to the lowest segment.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "fp16_bits_from_float64", "float64_from_fp16_bits",
    "gptq_perm_from_g_idx", "pack_gptq", "unpack_gptq_codes", "unpack_gptq_zeros",
    "dequant_gptq", "dequant_gptq_definitional",
    "exl2_seg_word_off", "pack_exl2", "unpack_exl2_codes", "dequant_exl2",
    "dequant_exl2_definitional", "pack_exl2_qscale", "unpack_exl2_qscale", "exl2_two_level_scales",
    "dequant_exl2_qscale", "matmul", "quantize_rtn", "EXL2_BITS", "SEGMENT_ROWS",
    "KV_BITS", "kv_quantize", "kv_pack", "kv_unpack", "kv_dequantize",
    "rtn_quantize_exl2", "rtn_errors_exl2", "solve_exl2_bits",
]

# ----------------------------------------------------------------------------
# fp16 (IEEE-754 binary16) encode / decode, written from the format definition
# ----------------------------------------------------------------------------

_F16_MAX = 65504.0          # (2 - 2^-10) * 2^15
_F16_OVERFLOW = 65520.0     # halfway between 65504 and 2^16: ties-to-even goes to inf
_F16_EMIN = -14
_F16_SUBNORMAL_QUANTUM = 2.0 ** -24


def fp16_bits_from_float64(v) -> np.ndarray:
    """Round float64 values to binary16 with round-to-nearest, ties to even.

    Returns the uint16 bit patterns. Subnormals are produced (no flush to
    zero), values at or above 65520 in magnitude become infinity, the sign of
    zero is kept and NaN becomes the quiet NaN 0x7E00 with its sign.
    """
    v = np.asarray(v, dtype=np.float64)
    sign = np.signbit(v).astype(np.uint16) << 15
    a = np.abs(v)
    out = np.zeros(v.shape, dtype=np.uint16)

    nan = np.isnan(a)
    inf = ~nan & (a >= _F16_OVERFLOW)
    fin = ~nan & ~inf

    # exponent of the leading bit: a = m * 2^E, m in [0.5, 1)  ->  e = E - 1
    _, E = np.frexp(np.where(fin & (a > 0), a, 1.0))
    e = E.astype(np.int64) - 1

    sub = fin & ((e < _F16_EMIN) | (a == 0))
    nrm = fin & ~sub

    # subnormal range: integer multiple of 2^-24, round half to even
    n_sub = np.rint(np.where(sub, a, 0.0) / _F16_SUBNORMAL_QUANTUM)
    # (n_sub may reach 1024 = the smallest normal; its bit pattern is the same)
    out = np.where(sub, n_sub.astype(np.uint16), out)

    # normal range: 11-bit significand n in [1024, 2048), quantum 2^(e-10)
    en = np.where(nrm, e, 0)
    n_nrm = np.rint(np.where(nrm, a, 1.0) / np.exp2((en - 10).astype(np.float64)))
    carry = n_nrm >= 2048
    en = np.where(carry, en + 1, en)
    n_nrm = np.where(carry, 1024.0, n_nrm)
    bits_nrm = (((en + 15).astype(np.int64) << 10) | (n_nrm.astype(np.int64) - 1024)).astype(np.uint16)
    out = np.where(nrm, bits_nrm, out)

    out = np.where(inf, np.uint16(0x7C00), out)
    out = np.where(nan, np.uint16(0x7E00), out)
    return (out | sign).astype(np.uint16)


def float64_from_fp16_bits(h) -> np.ndarray:
    """Exact value of binary16 bit patterns, decoded field by field."""
    h = np.asarray(h, dtype=np.uint16).astype(np.int64)
    s = np.where(h & 0x8000, -1.0, 1.0)
    ex = (h >> 10) & 0x1F
    fr = (h & 0x3FF).astype(np.float64)
    val = np.where(ex == 0, fr * _F16_SUBNORMAL_QUANTUM,
                   (1024.0 + fr) * np.exp2((ex - 25).astype(np.float64)))
    val = np.where(ex == 31, np.where(fr == 0, np.inf, np.nan), val)
    return s * val


def _as_f64(s_fp16) -> np.ndarray:
    """fp16 array (numpy float16 or uint16 bits) -> exact float64."""
    s_fp16 = np.asarray(s_fp16)
    if s_fp16.dtype == np.float16:
        s_fp16 = s_fp16.view(np.uint16)
    return float64_from_fp16_bits(s_fp16)


# ----------------------------------------------------------------------------
# GPTQ: 4-bit codes, per-group fp16 scale and 4-bit zero, optional act-order
# ----------------------------------------------------------------------------

def gptq_perm_from_g_idx(g_idx, group_size: int) -> np.ndarray:
    """Stored-row order for act-order: rows sorted stably by (g_idx[k], k).

    ``perm[j]`` is the original row held by stored row j, so stored rows
    ``[g*gs, (g+1)*gs)`` are exactly the rows of group g.
    """
    g_idx = np.asarray(g_idx, dtype=np.int64)
    K = g_idx.size
    if K % group_size:
        raise ValueError("K must be a multiple of group_size")
    counts = np.bincount(g_idx, minlength=K // group_size)
    if counts.size != K // group_size or np.any(counts != group_size) or g_idx.min() < 0:
        raise ValueError("every group must hold exactly group_size rows")
    return np.argsort(g_idx, kind="stable").astype(np.int32)


def pack_gptq(q, z, s, g_idx, group_size: int):
    """Pack an unpacked GPTQ layer, one bit at a time.

    q uint8 [K, N] (original row order), z uint8 [G, N], s fp16 [G, N],
    g_idx [K] (None = k // group_size).
    Returns (qweight uint32 [K/8, N], qzeros uint32 [G, N/8],
    scales uint16 [G, N] (fp16 bits), perm int32 [K]).
    Stored row j = 8r + i sits in nibble i (bits 4i..4i+3) of qweight[r];
    zero of column n = 8c + i sits in nibble i of qzeros[g][c].
    """
    q = np.asarray(q, dtype=np.uint8)
    K, N = q.shape
    if K % 8 or N % 8:
        raise ValueError("K and N must be multiples of 8")
    if g_idx is None:
        g_idx = np.arange(K) // group_size
    perm = gptq_perm_from_g_idx(g_idx, group_size)
    q_st = q[perm]
    qweight = np.zeros((K // 8, N), dtype=np.uint32)
    for i in range(8):
        for t in range(4):
            bit = ((q_st[i::8] >> t) & 1).astype(np.uint32)
            qweight |= bit << np.uint32(4 * i + t)
    z = np.asarray(z, dtype=np.uint8)
    G = z.shape[0]
    qzeros = np.zeros((G, N // 8), dtype=np.uint32)
    for i in range(8):
        for t in range(4):
            bit = ((z[:, i::8] >> t) & 1).astype(np.uint32)
            qzeros |= bit << np.uint32(4 * i + t)
    scales = np.asarray(s).view(np.uint16).copy() if np.asarray(s).dtype == np.float16 else np.asarray(s, dtype=np.uint16).copy()
    return qweight, qzeros, scales, perm


def unpack_gptq_codes(qweight, K: int) -> np.ndarray:
    """uint8 [K, N] codes in stored-row order, read back one bit at a time."""
    qweight = np.asarray(qweight, dtype=np.uint32)
    N = qweight.shape[1]
    q = np.zeros((K, N), dtype=np.uint8)
    for j in range(8):
        for t in range(4):
            bit = ((qweight >> np.uint32(4 * j + t)) & np.uint32(1)).astype(np.uint8)
            q[j::8] |= bit << t
    return q


def unpack_gptq_zeros(qzeros, N: int) -> np.ndarray:
    """uint8 [G, N] zero points, read back one bit at a time."""
    qzeros = np.asarray(qzeros, dtype=np.uint32)
    G = qzeros.shape[0]
    z = np.zeros((G, N), dtype=np.uint8)
    for i in range(8):
        for t in range(4):
            bit = ((qzeros >> np.uint32(4 * i + t)) & np.uint32(1)).astype(np.uint8)
            z[:, i::8] |= bit << t
    return z


def _scatter_rows(W_st: np.ndarray, perm) -> np.ndarray:
    if perm is None:
        return W_st
    W = np.empty_like(W_st)
    W[np.asarray(perm, dtype=np.int64)] = W_st
    return W


def dequant_gptq(qweight, qzeros, scales, perm, K: int, group_size: int, cols=None) -> np.ndarray:
    """fp16 bit patterns of W [K, N'] in ORIGINAL row order from packed GPTQ.

    w(j, n) = fp16_RNE((q(j, n) - z(j // gs, n)) * s(j // gs, n)) for stored
    row j, then W[perm[j]] = w(j). ``cols`` selects a subset of columns (the
    result is the same as slicing the full W).
    """
    qweight = np.asarray(qweight, dtype=np.uint32)
    N = qweight.shape[1]
    z = unpack_gptq_zeros(qzeros, N)
    s = _as_f64(scales)
    if cols is not None:
        cols = np.asarray(cols, dtype=np.int64)
        qweight, z, s = qweight[:, cols], z[:, cols], s[:, cols]
    q = unpack_gptq_codes(qweight, K)
    g = np.arange(K) // group_size
    w = (q.astype(np.int64) - z[g].astype(np.int64)).astype(np.float64) * s[g]
    return _scatter_rows(fp16_bits_from_float64(w), perm)


def dequant_gptq_definitional(q, z, s, g_idx, group_size: int) -> np.ndarray:
    """W [K, N] fp16 bits straight from the unpacked inputs (no packing):
    W[k][n] = fp16_RNE((q[k][n] - z[g_idx[k]][n]) * s[g_idx[k]][n])."""
    q = np.asarray(q)
    K = q.shape[0]
    if g_idx is None:
        g_idx = np.arange(K) // group_size
    g = np.asarray(g_idx, dtype=np.int64)
    s64 = _as_f64(s)
    w = (q.astype(np.int64) - np.asarray(z, dtype=np.int64)[g]).astype(np.float64) * s64[g]
    return fp16_bits_from_float64(w)


# ----------------------------------------------------------------------------
# EXL2: 32-row segments at 2/3/4/5/6/8 bits, symmetric, row permutation
# ----------------------------------------------------------------------------

SEGMENT_ROWS = 32
EXL2_BITS = (2, 3, 4, 5, 6, 8)


def exl2_seg_word_off(bits) -> np.ndarray:
    """uint32 [S+1]: first word row of each segment (prefix sums of bits)."""
    bits = np.asarray(bits, dtype=np.int64)
    off = np.zeros(bits.size + 1, dtype=np.int64)
    off[1:] = np.cumsum(bits)
    return off.astype(np.uint32)


def pack_exl2(q_st, bits, s, perm):
    """Pack an unpacked EXL2 layer one bit at a time.

    q_st uint8 [K, N] in stored order, bits [S], s fp16 [S, N], perm [K] or
    None. Returns (qweight uint32 [sum(bits), N], seg_word_off uint32 [S+1],
    scales uint16 [S, N], perm int32 [K] or None).
    """
    q_st = np.asarray(q_st, dtype=np.uint8)
    K, N = q_st.shape
    bits = np.asarray(bits, dtype=np.int64)
    if K % SEGMENT_ROWS or bits.size != K // SEGMENT_ROWS:
        raise ValueError("K must be 32 * len(bits)")
    if not set(bits.tolist()) <= set(EXL2_BITS):
        raise ValueError("bit widths must be in {2,3,4,5,6,8}")
    off = exl2_seg_word_off(bits).astype(np.int64)
    qweight = np.zeros((int(off[-1]), N), dtype=np.uint32)
    for b in np.unique(bits):
        segs = np.flatnonzero(bits == b)
        for i in range(SEGMENT_ROWS):
            codes = q_st[segs * SEGMENT_ROWS + i]            # [len(segs), N]
            for t in range(int(b)):
                p = i * int(b) + t                            # stream bit position
                bit = ((codes >> t) & 1).astype(np.uint32)
                qweight[off[segs] + p // 32] |= bit << np.uint32(p % 32)
    sc = np.asarray(s)
    sc = sc.view(np.uint16).copy() if sc.dtype == np.float16 else sc.astype(np.uint16)
    return qweight, off.astype(np.uint32), sc, (None if perm is None else np.asarray(perm, dtype=np.int32))


def unpack_exl2_codes(qweight, bits, seg_word_off=None) -> np.ndarray:
    """uint8 [K, N] codes in stored order, read back one stream bit at a time."""
    qweight = np.asarray(qweight, dtype=np.uint32)
    bits = np.asarray(bits, dtype=np.int64)
    off = (exl2_seg_word_off(bits) if seg_word_off is None else np.asarray(seg_word_off)).astype(np.int64)
    K, N = bits.size * SEGMENT_ROWS, qweight.shape[1]
    q = np.zeros((K, N), dtype=np.uint8)
    for b in np.unique(bits):
        segs = np.flatnonzero(bits == b)
        for i in range(SEGMENT_ROWS):
            for t in range(int(b)):
                p = i * int(b) + t
                word = qweight[off[segs] + p // 32]
                bit = ((word >> np.uint32(p % 32)) & np.uint32(1)).astype(np.uint8)
                q[segs * SEGMENT_ROWS + i] |= bit << t
    return q


def dequant_exl2(qweight, seg_word_off, bits, scales, perm, cols=None) -> np.ndarray:
    """fp16 bits of W [K, N'] in ORIGINAL row order from packed EXL2.

    w(j, n) = fp16_RNE((q(j, n) - 2^(b-1)) * s(j // 32, n)) with b the width
    of segment j // 32, then W[perm[j]] = w(j).
    """
    qweight = np.asarray(qweight, dtype=np.uint32)
    s = _as_f64(scales)
    if cols is not None:
        cols = np.asarray(cols, dtype=np.int64)
        qweight, s = qweight[:, cols], s[:, cols]
    bits = np.asarray(bits, dtype=np.int64)
    q = unpack_exl2_codes(qweight, bits, seg_word_off)
    seg = np.arange(q.shape[0]) // SEGMENT_ROWS
    z = (1 << (bits[seg] - 1)).astype(np.int64)
    w = (q.astype(np.int64) - z[:, None]).astype(np.float64) * s[seg]
    return _scatter_rows(fp16_bits_from_float64(w), perm)


def dequant_exl2_definitional(q_st, bits, s, perm) -> np.ndarray:
    """W [K, N] fp16 bits straight from the unpacked inputs (no packing)."""
    q_st = np.asarray(q_st)
    bits = np.asarray(bits, dtype=np.int64)
    seg = np.arange(q_st.shape[0]) // SEGMENT_ROWS
    z = (1 << (bits[seg] - 1)).astype(np.int64)
    w = (q_st.astype(np.int64) - z[:, None]).astype(np.float64) * _as_f64(s)[seg]
    return _scatter_rows(fp16_bits_from_float64(w), perm)


# ----------------------------------------------------------------------------
# EXL2 with two-level scales (4-bit group scale code x per-column maximum)
# ----------------------------------------------------------------------------

def pack_exl2_qscale(codes) -> np.ndarray:
    """uint8 [S, N] codes 0..15 -> uint32 [S, N/8], one bit at a time:
    bit t of column n = 8k + i goes to bit 4i + t of word k."""
    codes = np.asarray(codes, dtype=np.uint8)
    S, N = codes.shape
    if N % 8 or (codes > 15).any():
        raise ValueError("N must be a multiple of 8 and codes below 16")
    out = np.zeros((S, N // 8), dtype=np.uint32)
    for n in range(N):
        k, i = divmod(n, 8)
        for t in range(4):
            bit = ((codes[:, n] >> t) & 1).astype(np.uint32)
            out[:, k] |= bit << np.uint32(4 * i + t)
    return out


def unpack_exl2_qscale(words, N: int) -> np.ndarray:
    """uint32 [S, N/8] -> uint8 [S, N] codes, one bit at a time."""
    words = np.asarray(words, dtype=np.uint32)
    out = np.zeros((words.shape[0], N), dtype=np.uint8)
    for n in range(N):
        k, i = divmod(n, 8)
        for t in range(4):
            bit = ((words[:, k] >> np.uint32(4 * i + t)) & np.uint32(1)).astype(np.uint8)
            out[:, n] |= bit << t
    return out


def exl2_two_level_scales(codes, scale_max) -> np.ndarray:
    """Exact float64 values [S, N] of s(g, n) = ((c(g, n) + 1) / 16) * m(n).

    codes uint8 [S, N] (0..15), scale_max fp16 [N]. Not rounded: the
    product has at most 5 + 11 significant bits, so float64 holds it."""
    c = np.asarray(codes, dtype=np.int64)
    m = _as_f64(scale_max)
    frac = (c + 1).astype(np.float64) / 16.0        # exact: k / 16, k = 1..16
    return frac * m[None, :]


def dequant_exl2_qscale(qweight, seg_word_off, bits, q_scale, scale_max, perm, cols=None) -> np.ndarray:
    """fp16 bits of W [K, N'] in ORIGINAL row order from packed EXL2 with
    two-level scales: w(j, n) = fp16_RNE((q(j, n) - 2^(b-1)) * s(j // 32, n))
    with the exact scales of exl2_two_level_scales (one rounding: the float64
    product is exact), then W[perm[j]] = w(j)."""
    q_scale = np.asarray(q_scale, dtype=np.uint32)
    N = q_scale.shape[1] * 8
    bits = np.asarray(bits, dtype=np.int64)
    s = exl2_two_level_scales(unpack_exl2_qscale(q_scale, N), scale_max)
    if cols is not None:
        cols = np.asarray(cols, dtype=np.int64)
        qweight = np.asarray(qweight, dtype=np.uint32)[:, cols]
        s = s[:, cols]
    q = unpack_exl2_codes(qweight, bits, seg_word_off).astype(np.int64)
    seg = np.arange(q.shape[0]) // SEGMENT_ROWS
    z = (np.int64(1) << (bits[seg] - 1))[:, None]
    w = (q - z).astype(np.float64) * s[seg]
    return _scatter_rows(fp16_bits_from_float64(w), perm)


# ----------------------------------------------------------------------------
# Quantized KV cache codec (Q4 / Q6 / Q8)
# ----------------------------------------------------------------------------

KV_BITS = (4, 6, 8)


def kv_quantize(x, b: int):
    """fp16 x [G, D] (numpy float16 or uint16 bits) -> (codes uint8 [G, D],
    scales uint16 fp16 bits [G]); the steps of the codec reading above."""
    if b not in KV_BITS:
        raise ValueError("b must be 4, 6 or 8")
    x32 = _as_f64(x).astype(np.float32)                  # exact: fp16 values are fp32 values
    qmax = (1 << (b - 1)) - 1
    amax = np.abs(x32).max(axis=1)
    s32 = amax / np.float32(qmax)                        # IEEE fp32 division, round to nearest even
    s_bits = fp16_bits_from_float64(s32.astype(np.float64))
    s = float64_from_fp16_bits(s_bits).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = x32 / s[:, None]                             # fp32 quotient
    q = np.where(s[:, None] == 0, np.float32(0), np.rint(r))
    q = np.clip(q, -qmax - 1, qmax).astype(np.int64)
    return (q + (1 << (b - 1))).astype(np.uint8), s_bits


def kv_pack(codes, b: int) -> np.ndarray:
    """uint8 codes [G, D] -> uint32 [G, D*b/32]: code i of a group at bits
    [i*b, i*b+b) of its word stream, one bit at a time."""
    codes = np.asarray(codes, dtype=np.uint8)
    G, D = codes.shape
    if (D * b) % 32:
        raise ValueError("D * b must be a multiple of 32")
    out = np.zeros((G, D * b // 32), dtype=np.uint32)
    for i in range(D):
        for t in range(b):
            p = i * b + t
            bit = ((codes[:, i] >> t) & 1).astype(np.uint32)
            out[:, p // 32] |= bit << np.uint32(p % 32)
    return out


def kv_unpack(words, b: int, D: int) -> np.ndarray:
    """uint32 [G, D*b/32] -> uint8 codes [G, D], one bit at a time."""
    words = np.asarray(words, dtype=np.uint32)
    out = np.zeros((words.shape[0], D), dtype=np.uint8)
    for i in range(D):
        for t in range(b):
            p = i * b + t
            bit = ((words[:, p // 32] >> np.uint32(p % 32)) & np.uint32(1)).astype(np.uint8)
            out[:, i] |= bit << t
    return out


def kv_dequantize(words, scales, b: int, D: int) -> np.ndarray:
    """fp16 bits [G, D] of fp16_RNE((u - 2^(b-1)) * s); the product is exact
    in float64."""
    u = kv_unpack(words, b, D).astype(np.int64) - (1 << (b - 1))
    return fp16_bits_from_float64(u.astype(np.float64) * _as_f64(scales)[:, None])


# ----------------------------------------------------------------------------
# EXL2 conversion: RTN quantizer, weight-space error table, bits solve
# ----------------------------------------------------------------------------

def _rtn_columns(v32, b: int):
    """Symmetric RTN of groups along axis 0 (fp32 values): the KV codec's
    arithmetic. Returns (codes uint8, scale fp16 bits per column)."""
    qmax = (1 << (b - 1)) - 1
    amax = np.abs(v32).max(axis=0)
    s_bits = fp16_bits_from_float64((amax / np.float32(qmax)).astype(np.float64))
    s = float64_from_fp16_bits(s_bits).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = v32 / s[None, :]
    q = np.where(s[None, :] == 0, np.float32(0), np.rint(r))
    q = np.clip(q, -qmax - 1, qmax).astype(np.int64)
    return (q + (1 << (b - 1))).astype(np.uint8), s_bits


def rtn_quantize_exl2(W, perm, bits):
    """fp16 W [K, N] in input-feature order, perm [K] (stored row j = input
    row perm[j]) or None, widths [S] -> (codes uint8 [K, N] in stored order,
    scales uint16 fp16 bits [S, N]) ready for pack_exl2."""
    Wv = _as_f64(W)
    if perm is not None:
        Wv = Wv[np.asarray(perm, dtype=np.int64)]
    bits = np.asarray(bits, dtype=np.int64)
    K, N = Wv.shape
    q = np.zeros((K, N), dtype=np.uint8)
    s = np.zeros((bits.size, N), dtype=np.uint16)
    for seg, b in enumerate(bits):
        rows = slice(seg * SEGMENT_ROWS, (seg + 1) * SEGMENT_ROWS)
        q[rows], s[seg] = _rtn_columns(Wv[rows].astype(np.float32), int(b))
    return q, s


def rtn_errors_exl2(W, perm) -> np.ndarray:
    """float64 [S, 6]: sum over the segment's 32 x N weights of (w - w_hat)^2
    at each width of EXL2_BITS, w_hat the fp16 dequantisation of the RTN codes."""
    Wv = _as_f64(W)
    if perm is not None:
        Wv = Wv[np.asarray(perm, dtype=np.int64)]
    S = Wv.shape[0] // SEGMENT_ROWS
    err = np.zeros((S, len(EXL2_BITS)), dtype=np.float64)
    for seg in range(S):
        v = Wv[seg * SEGMENT_ROWS:(seg + 1) * SEGMENT_ROWS]
        for i, b in enumerate(EXL2_BITS):
            u, s_bits = _rtn_columns(v.astype(np.float32), b)
            w_hat = float64_from_fp16_bits(fp16_bits_from_float64(
                (u.astype(np.int64) - (1 << (b - 1))).astype(np.float64) * float64_from_fp16_bits(s_bits)[None, :]))
            err[seg, i] = np.sum((v - w_hat) ** 2)
    return err


def solve_exl2_bits(err, budget: int) -> np.ndarray:
    """Widths [S] from the error table [S, 6] and a budget of total code bits
    per column (sum of widths): every segment starts at 2 bits; while some
    step to the next width fits the budget, take the one with the largest
    (err[b] - err[b_next]) / (b_next - b), the lowest segment on ties."""
    err = np.asarray(err, dtype=np.float64)
    S = err.shape[0]
    level = np.zeros(S, dtype=np.int64)          # index into EXL2_BITS
    widths = np.array(EXL2_BITS, dtype=np.int64)
    total = 2 * S
    if budget < total:
        raise ValueError("budget below two bits per segment")
    while True:
        best, best_gain = -1, None
        for seg in range(S):
            lv = level[seg]
            if lv + 1 >= len(widths):
                continue
            step = int(widths[lv + 1] - widths[lv])
            if total + step > budget:
                continue
            gain = (err[seg, lv] - err[seg, lv + 1]) / step
            if best_gain is None or gain > best_gain:
                best, best_gain = seg, gain
        if best < 0:
            break
        total += int(widths[level[best] + 1] - widths[level[best]])
        level[best] += 1
    return widths[level].astype(np.uint8)


# ----------------------------------------------------------------------------
# Matmul and the round-trip quantizer
# ----------------------------------------------------------------------------

def matmul(x, W_bits) -> np.ndarray:
    """y [M, N] = x [M, K] . W [K, N] accumulated in float64.

    x is fp16 (numpy float16 or uint16 bits), W_bits uint16 fp16 bits.
    """
    return np.matmul(_as_f64(x), float64_from_fp16_bits(W_bits))


def quantize_rtn(W_bits, s, z, b: int) -> np.ndarray:
    """Round-to-nearest quantizer used for round-trip checks:
    q = clamp(rint(W / s) + z, 0, 2^b - 1) (ties to even)."""
    W = float64_from_fp16_bits(W_bits)
    q = np.rint(W / _as_f64(s)) + np.asarray(z, dtype=np.float64)
    return np.clip(q, 0, (1 << b) - 1).astype(np.uint8)
