"""Pins for the CPU oracle: each check fixes the oracle against something other
than itself (hand-derived fixtures, numpy's and Python's own float16
conversions, exact integer / rational arithmetic, one-hot inputs, permutation
invariance, a cross-format reduction, big-integer bit streams)."""
from __future__ import annotations

import struct
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = Path(__file__).parent / "golden"


def _fixture(name):
    rows = []
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.split("#", 1)[0].strip()
        if line:
            rows.append(line)
    return rows


def _py_half_bits(v: float) -> int:
    """Python's own binary16 conversion (struct 'e', round-half-even)."""
    try:
        return struct.unpack("<H", struct.pack("<e", v))[0]
    except OverflowError:
        return 0xFC00 if v < 0 else 0x7C00


# ---------------------------------------------------------------- fp16 rounding

def test_fp16_rounding_golden():
    for row in _fixture("fp16_rounding.txt"):
        expr, want = row.rsplit(None, 1)
        v = float(eval(expr, {}, {}))
        got = int(O.fp16_bits_from_float64(np.array([v]))[0])
        assert got == int(want, 16), (expr, hex(got), want)


def test_fp16_rounding_matches_numpy_random():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(400_000) * np.exp2(rng.integers(-30, 18, 400_000))
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(O.fp16_bits_from_float64(x), want)


def test_fp16_rounding_every_tie_and_neighbour():
    # every fp16 value h, the exact midpoints to its neighbour, and points just
    # beside them, in every binade including subnormals: compare with numpy and
    # Python's struct 'e' (both correctly rounded)
    h = np.arange(0, 0x7C00, dtype=np.uint16)
    v = O.float64_from_fp16_bits(h)
    nxt = O.float64_from_fp16_bits(h + 1) if True else None
    mid = (v + nxt) / 2.0
    cands = np.concatenate([v, mid, np.nextafter(mid, 0), np.nextafter(mid, np.inf)])
    cands = np.concatenate([cands, -cands])
    with np.errstate(over="ignore"):
        want = cands.astype(np.float16).view(np.uint16)
    got = O.fp16_bits_from_float64(cands)
    assert np.array_equal(got, want)
    sample = cands[:: 997]
    assert [int(b) for b in O.fp16_bits_from_float64(sample)] == [_py_half_bits(float(c)) for c in sample]


def test_fp16_decode_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = O.float64_from_fp16_bits(h)
    want = h.view(np.float16).astype(np.float64)
    fin = np.isfinite(want)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    assert np.array_equal(got[fin], want[fin])
    assert np.array_equal(np.signbit(got[fin]), np.signbit(want[fin]))
    assert np.array_equal(got[np.isinf(want)], want[np.isinf(want)])


# ---------------------------------------------------------------- GPTQ layout

def test_gptq_golden_words():
    for row in _fixture("gptq_words.txt"):
        tok = row.split()
        word, zero, scale = int(tok[0], 16), int(tok[1]), int(tok[2], 16)
        want = [int(t, 16) for t in tok[3:]]
        K = N = 8
        qweight = np.zeros((1, N), dtype=np.uint32)
        qweight[0, 0] = word
        qzeros = np.zeros((1, 1), dtype=np.uint32)
        qzeros[0, 0] = zero            # nibble 0 = zero of column 0
        scales = np.zeros((1, N), dtype=np.uint16)
        scales[0, 0] = scale
        W = O.dequant_gptq(qweight, qzeros, scales, None, K, 8)
        assert [int(v) for v in W[:, 0]] == want, tok[0]


def test_gptq_zero_nibbles():
    # zero of column n = 8c + i lives in nibble i of qzeros[g][c]
    N = 16
    qz = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    assert O.unpack_gptq_zeros(qz, N)[0].tolist() == list(range(16))


@pytest.mark.parametrize("act_order", [False, True])
def test_gptq_roundtrip_and_definitional(act_order):
    inp = synth.gptq_layer(256, 48, group_size=32, act_order=act_order, seed=3)
    qw, qz, sc, perm = O.pack_gptq(inp.q, inp.z, inp.s, inp.g_idx, 32)
    assert np.array_equal(O.unpack_gptq_codes(qw, 256), inp.q[perm])
    assert np.array_equal(O.unpack_gptq_zeros(qz, 48), inp.z)
    # stored rows of group g are the rows of group g
    assert np.array_equal(inp.g_idx[perm], np.arange(256) // 32)
    W_packed = O.dequant_gptq(qw, qz, sc, perm, 256, 32)
    W_def = O.dequant_gptq_definitional(inp.q, inp.z, inp.s, inp.g_idx, 32)
    assert np.array_equal(W_packed, W_def)
    cols = np.array([0, 5, 17, 47])
    assert np.array_equal(O.dequant_gptq(qw, qz, sc, perm, 256, 32, cols=cols), W_def[:, cols])


def test_gptq_adversarial_codes_roundtrip():
    K, N = 64, 16
    for q in (np.full((K, N), 15, np.uint8), np.zeros((K, N), np.uint8),
              (np.indices((K, N)).sum(0) % 2 * 15).astype(np.uint8),
              np.tile(np.array([5, 10], np.uint8), (K, N // 2))):
        z = np.full((K // 8, N), 7, np.uint8)
        s = np.full((K // 8, N), 1.0, np.float16)
        qw, qz, _, perm = O.pack_gptq(q, z, s, None, 8)
        assert np.array_equal(perm, np.arange(K))
        assert np.array_equal(O.unpack_gptq_codes(qw, K), q)


def test_gptq_stable_sort_tie_break():
    g_idx = np.array([1, 0, 1, 0, 1, 0, 1, 0] * 2)
    perm = O.gptq_perm_from_g_idx(g_idx, 8)
    assert perm.tolist() == [1, 3, 5, 7, 9, 11, 13, 15, 0, 2, 4, 6, 8, 10, 12, 14]
    with pytest.raises(ValueError):
        O.gptq_perm_from_g_idx(np.array([0] * 9 + [1] * 7), 8)


# ---------------------------------------------------------------- EXL2 layout

def _pattern(spec: str, b: int):
    i = np.arange(32)
    if spec.startswith("imod"):
        return i % int(spec[4:])
    if spec == "i":
        return i.copy()
    pos, val = spec[1:].split("=")
    out = np.zeros(32, dtype=np.int64)
    out[int(pos)] = int(val)
    return out


def test_exl2_golden_streams():
    for row in _fixture("exl2_streams.txt"):
        tok = row.split()
        b, spec, words = int(tok[0]), tok[1], [int(t, 16) for t in tok[2:]]
        codes = _pattern(spec, b).astype(np.uint8)
        q_st = np.zeros((32, 8), dtype=np.uint8)
        q_st[:, 3] = codes
        qw, off, _, _ = O.pack_exl2(q_st, [b], np.ones((1, 8), np.float16), None)
        assert off.tolist() == [0, b]
        assert [int(w) for w in qw[:, 3]] == words, (b, spec)
        assert not qw[:, [0, 1, 2, 4, 5, 6, 7]].any()
        assert np.array_equal(O.unpack_exl2_codes(qw, [b])[:, 3], codes)


def test_exl2_every_value_at_every_position():
    # brute force: code v at position i of a segment occupies stream bits
    # [i*b, i*b+b) as the bits of v; built here as one Python big integer
    for b in O.EXL2_BITS:
        for i in range(32):
            for v in {1, (1 << b) - 1, (1 << b) >> 1, 0b101 & ((1 << b) - 1)}:
                q_st = np.zeros((32, 8), dtype=np.uint8)
                q_st[i, 0] = v
                qw, _, _, _ = O.pack_exl2(q_st, [b], np.ones((1, 8), np.float16), None)
                stream = v << (i * b)
                want = [(stream >> (32 * t)) & 0xFFFFFFFF for t in range(b)]
                assert [int(w) for w in qw[:, 0]] == want, (b, i, v)
                assert int(O.unpack_exl2_codes(qw, [b])[i, 0]) == v


def test_exl2_roundtrip_and_definitional():
    inp = synth.exl2_layer(512, 40, bpw=4.0, seed=5)
    qw, off, sc, perm = O.pack_exl2(inp.q, inp.bits, inp.s, inp.perm)
    assert off[-1] == int(inp.bits.astype(int).sum()) == 4 * 16
    assert np.array_equal(O.unpack_exl2_codes(qw, inp.bits, off), inp.q)
    W_packed = O.dequant_exl2(qw, off, inp.bits, sc, perm)
    W_def = O.dequant_exl2_definitional(inp.q, inp.bits, inp.s, inp.perm)
    assert np.array_equal(W_packed, W_def)
    cols = np.array([1, 7, 39])
    assert np.array_equal(O.dequant_exl2(qw, off, inp.bits, sc, perm, cols=cols), W_def[:, cols])


def test_exl2_big_integer_packing_random():
    # the whole packed tensor rebuilt with Python big integers, per column
    inp = synth.exl2_layer(32 * 6, 8, bits=np.array([2, 3, 4, 5, 6, 8]), seed=9)
    qw, off, _, _ = O.pack_exl2(inp.q, inp.bits, inp.s, None)
    for n in range(8):
        col = []
        for s_, b in enumerate(inp.bits.tolist()):
            stream = 0
            for i in range(32):
                stream |= int(inp.q[32 * s_ + i, n]) << (i * b)
            col += [(stream >> (32 * t)) & 0xFFFFFFFF for t in range(b)]
        assert [int(w) for w in qw[:, n]] == col


# ---------------------------------------------------------------- dequant

def test_dequant_exhaustive_vs_numpy():
    # every (q, z) pair of 4-bit codes and of 8-bit codes against a sweep of
    # scales (normal, subnormal-producing, overflowing, negative); reference =
    # numpy's float64 -> float16 cast of the exact product
    scales = np.array([0.005, 0.0123, 0.02, -0.0177, 2.0 ** -20, -(2.0 ** -24), 3.0 ** -9,
                       1000.0, 4100.0, -65504.0, 1.0 + 2.0 ** -10, 0.0, -0.0, 0.333], dtype=np.float64)
    s16 = scales.astype(np.float16)
    for nbits in (4, 8):
        qq, zz = np.meshgrid(np.arange(1 << nbits), np.arange(1 << nbits), indexing="ij")
        d = (qq - zz).reshape(-1, 1).astype(np.float64)
        prod = d * s16.astype(np.float64).reshape(1, -1)
        with np.errstate(over="ignore"):
            want = prod.astype(np.float16).view(np.uint16)
        got = O.fp16_bits_from_float64(prod)
        assert np.array_equal(got, want)


def test_dequant_exl2_zero_point_is_half_range():
    # a code equal to 2^(b-1) dequantises to +0 for every width; codes 0 and
    # 2^b - 1 give -2^(b-1)*s and (2^(b-1)-1)*s
    for b in O.EXL2_BITS:
        q_st = np.zeros((32, 8), dtype=np.uint8)
        q_st[0, :] = 1 << (b - 1)
        q_st[1, :] = (1 << b) - 1
        s = np.full((1, 8), 0.5, np.float16)
        qw, off, sc, _ = O.pack_exl2(q_st, [b], s, None)
        W = O.float64_from_fp16_bits(O.dequant_exl2(qw, off, [b], sc, None))
        assert np.all(W[0] == 0) and not np.signbit(W[0]).any()
        assert np.all(W[1] == ((1 << (b - 1)) - 1) * 0.5)
        assert np.all(W[2] == -(1 << (b - 1)) * 0.5)


def test_rtn_idempotence():
    # quantize(dequant(q)) == q: fp16 rounding moves w by at most 2^-11 |w|,
    # i.e. < 0.5 code steps for |q - z| <= 255
    inp = synth.gptq_layer(128, 32, group_size=32, seed=11)
    W = O.dequant_gptq_definitional(inp.q, inp.z, inp.s, None, 32)
    g = np.arange(128) // 32
    assert np.array_equal(O.quantize_rtn(W, inp.s[g], inp.z[g], 4), inp.q)
    e = synth.exl2_layer(128, 16, bits=np.array([8, 2, 6, 3]), permute=False, seed=12)
    W = O.dequant_exl2_definitional(e.q, e.bits, e.s, None)
    seg = np.arange(128) // 32
    z = (1 << (e.bits.astype(int)[seg] - 1))[:, None]
    for b in (8, 2, 6, 3):
        rows = np.flatnonzero(e.bits[seg] == b)
        assert np.array_equal(O.quantize_rtn(W[rows], e.s[seg][rows], z[rows], b), e.q[rows])


# ---------------------------------------------------------------- matmul

def _exact_int_y(x16, W_bits):
    """Exact y as Python integers in units of 2^-48 (fp16 values are
    multiples of 2^-24)."""
    xi = (O.float64_from_fp16_bits(np.asarray(x16).view(np.uint16)) * 2.0 ** 24).astype(np.int64)
    wi = (O.float64_from_fp16_bits(W_bits) * 2.0 ** 24).astype(np.int64)
    M, K = xi.shape
    N = wi.shape[1]
    y = [[0] * N for _ in range(M)]
    xl, wl = xi.tolist(), wi.tolist()
    for m in range(M):
        for k in range(K):
            a = xl[m][k]
            if a:
                row = wl[k]
                ym = y[m]
                for n in range(N):
                    ym[n] += a * row[n]
    return y


def test_matmul_vs_exact_integer():
    inp = synth.gptq_layer(128, 24, group_size=32, act_order=True, seed=21)
    qw, qz, sc, perm = O.pack_gptq(inp.q, inp.z, inp.s, inp.g_idx, 32)
    W = O.dequant_gptq(qw, qz, sc, perm, 128, 32)
    x = synth.activations(3, 128, seed=21)
    y = O.matmul(x, W)
    ye = _exact_int_y(x, W)
    for m in range(3):
        for n in range(24):
            exact = ye[m][n] / 2.0 ** 48
            assert abs(y[m, n] - exact) <= 1e-12 * max(1.0, abs(exact))


def test_one_hot_reproduces_rows():
    inp = synth.exl2_layer(96, 16, bits=np.array([3, 8, 5]), seed=31)
    qw, off, sc, perm = O.pack_exl2(inp.q, inp.bits, inp.s, inp.perm)
    W = O.dequant_exl2(qw, off, inp.bits, sc, perm)
    x = np.zeros((96, 96), dtype=np.float16)
    x[np.arange(96), np.arange(96)] = 1.0
    y = O.matmul(x, W)
    assert np.array_equal(y, O.float64_from_fp16_bits(W))
    # K != N so a transposed operand cannot pass
    assert y.shape == (96, 16)


def test_permutation_invariance_exact():
    # apply a random permutation pi to K of both x and W (composed into the
    # stored->original map): y must not change, exactly
    K, N, M = 160, 16, 2
    inp = synth.exl2_layer(K, N, bits=np.array([2, 4, 6, 8, 3]), seed=41)
    x = synth.activations(M, K, seed=41)
    qw, off, sc, perm = O.pack_exl2(inp.q, inp.bits, inp.s, inp.perm)
    W1 = O.dequant_exl2(qw, off, inp.bits, sc, perm)
    pi = np.random.default_rng(7).permutation(K)
    x2 = np.empty_like(x)
    x2[:, pi] = x
    perm2 = pi[perm]
    W2 = O.dequant_exl2(qw, off, inp.bits, sc, perm2)
    assert _exact_int_y(x, W1) == _exact_int_y(x2, W2)
    assert np.allclose(O.matmul(x, W1), O.matmul(x2, W2), rtol=1e-15, atol=1e-12)
    # and the same for GPTQ act-order: relabel the original rows
    g = synth.gptq_layer(K, N, group_size=32, act_order=True, seed=42)
    q2 = np.empty_like(g.q)
    q2[pi] = g.q
    gi2 = np.empty_like(g.g_idx)
    gi2[pi] = g.g_idx
    Wa = O.dequant_gptq(*O.pack_gptq(g.q, g.z, g.s, g.g_idx, 32)[:4], K, 32)
    Wb = O.dequant_gptq(*O.pack_gptq(q2, g.z, g.s, gi2, 32)[:4], K, 32)
    assert _exact_int_y(x, Wa) == _exact_int_y(x2, Wb)


def test_cross_format_exl2_4bit_is_gptq_gs32():
    # EXL2 with every segment at 4 bits and no permutation is GPTQ with group
    # size 32, every zero 8 and the same scales: same words, same weights
    K, N = 128, 16
    q = synth.gptq_layer(K, N, group_size=32, seed=51).q
    s = synth.fp16_uniform(np.random.default_rng(5), 0.002, 0.03, (K // 32, N))
    qw_e, off, sc_e, _ = O.pack_exl2(q, [4] * (K // 32), s, None)
    z = np.full((K // 32, N), 8, np.uint8)
    qw_g, qz_g, sc_g, perm = O.pack_gptq(q, z, s, None, 32)
    assert np.array_equal(qw_e, qw_g)
    assert np.array_equal(O.dequant_exl2(qw_e, off, [4] * (K // 32), sc_e, None),
                          O.dequant_gptq(qw_g, qz_g, sc_g, perm, K, 32))


def _brute_force_y(x16, Wfun, M, K, N):
    out = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += Fraction(float(x16[m, k])) * Fraction(Wfun(k, n))
            out[m, n] = float(acc)
    return out


def test_brute_force_gptq_8x8_tile():
    # 8x8 GPTQ tile with group size 8, act-order: weights by the definition in
    # pure Python (Python's own half conversion), y by exact rationals
    K = N = 8
    rng = np.random.default_rng(61)
    q = rng.integers(0, 16, (K, N)).astype(np.uint8)
    z = rng.integers(0, 16, (1, N)).astype(np.uint8)
    s = synth.fp16_uniform(rng, -0.02, 0.02, (1, N))
    x = synth.activations(2, K, seed=61)
    qw, qz, sc, perm = O.pack_gptq(q, z, s, None, 8)
    y = O.matmul(x, O.dequant_gptq(qw, qz, sc, perm, K, 8))

    def w(k, n):
        h = _py_half_bits((int(q[k, n]) - int(z[0, n])) * float(s[0, n]))
        return struct.unpack("<e", struct.pack("<H", h))[0]
    assert np.allclose(y, _brute_force_y(x, w, 2, K, N), rtol=1e-13, atol=0)


def test_brute_force_exl2_32x8_tile():
    for b in (3, 5, 6):
        rng = np.random.default_rng(70 + b)
        q = rng.integers(0, 1 << b, (32, 8)).astype(np.uint8)
        s = synth.fp16_uniform(rng, 0.002, 0.03, (1, 8))
        perm = rng.permutation(32).astype(np.int32)
        x = synth.activations(1, 32, seed=b)
        qw, off, sc, p = O.pack_exl2(q, [b], s, perm)
        y = O.matmul(x, O.dequant_exl2(qw, off, [b], sc, p))
        inv = np.argsort(perm)                       # original row k -> stored row

        def w(k, n):
            j = inv[k]
            h = _py_half_bits((int(q[j, n]) - (1 << (b - 1))) * float(s[0, n]))
            return struct.unpack("<e", struct.pack("<H", h))[0]
        assert np.allclose(y, _brute_force_y(x, w, 1, 32, 8), rtol=1e-13, atol=0)


# ---------------------------------------------------------------- shards

def test_shard_reductions():
    # column-parallel shards concatenate, row-parallel shards (on segment
    # boundaries) sum, to the unsharded result
    inp = synth.exl2_layer(256, 32, bpw=4.0, seed=81, permute=False)
    x = synth.activations(2, 256, seed=81)
    qw, off, sc, _ = O.pack_exl2(inp.q, inp.bits, inp.s, None)
    W = O.dequant_exl2(qw, off, inp.bits, sc, None)
    y = O.matmul(x, W)
    cat = np.concatenate([O.matmul(x, O.dequant_exl2(qw, off, inp.bits, sc, None, cols=np.arange(c, c + 16)))
                          for c in (0, 16)], axis=1)
    assert np.array_equal(cat, y)
    ks = []
    for lo, hi in ((0, 4), (4, 8)):
        o2 = off[lo:hi + 1] - off[lo]
        Wk = O.dequant_exl2(qw[off[lo]:off[hi]], o2, inp.bits[lo:hi], sc[lo:hi], None)
        ks.append(O.matmul(x[:, lo * 32:hi * 32], Wk))
    assert np.allclose(ks[0] + ks[1], y, rtol=1e-14, atol=1e-12)


# ---------------------------------------------------------------- generator

def test_bit_mix_is_exact():
    for S, bpw, allowed in ((128, 4.0, synth.EXL2_BITS), (344, 4.0, synth.EXL2_BITS),
                            (256, 2.5, (2, 3, 4)), (896, 2.5, (2, 3, 4))):
        bits = synth.solve_bit_mix(S, bpw, allowed, np.random.default_rng(S))
        assert int(bits.astype(int).sum()) == int(bpw * S)
        assert set(np.unique(bits).tolist()) <= set(allowed)


# ---------------------------------------------------------------- EXL2 two-level scales

def _qscale_weight(m_bits: int, c: int, v: int) -> int:
    """The oracle's dequantised weight for one (m, c, v = q - 128) through a
    one-segment, eight-column EXL2 layer of width 8 (packed by the oracle)."""
    q = np.full((32, 8), 128, dtype=np.uint8)
    q[0, 0] = v + 128
    bits = np.array([8])
    qw, off, _, _ = O.pack_exl2(q, bits, np.ones((1, 8), np.float16), None)
    codes = np.zeros((1, 8), np.uint8)
    codes[0, 0] = c
    m = np.full(8, m_bits, dtype=np.uint16)
    return int(O.dequant_exl2_qscale(qw, off, bits, O.pack_exl2_qscale(codes), m, None)[0, 0])


def test_exl2_qscale_golden():
    # hand-derived weights, including cases where rounding the scale to fp16
    # first would give another weight, ties, subnormals, -0 and overflow
    for row in _fixture("exl2_qscale.txt"):
        m_hex, c, v, want = row.split()
        got = _qscale_weight(int(m_hex, 16), int(c), int(v))
        assert got == int(want, 16), (m_hex, c, v, hex(got), want)


def test_exl2_qscale_matches_exact_rational_rounding():
    # every code, several values of q - z, against every fp16 maximum of a few
    # binades (normal and subnormal, both signs): the exact rational
    # v * (c + 1) / 16 * m rounded once by Python's own binary16 conversion
    # (struct 'e'; the float64 it starts from holds the rational exactly)
    hs = np.concatenate([np.arange(0x0000, 0x0800, 37), np.arange(0x2C00, 0x3C00, 53), np.arange(0x5000, 0x5800, 41),
                         np.arange(0x8001, 0x8400, 67)]).astype(np.uint16)
    vs = np.array([-128, -77, -8, -3, -1, 0, 1, 3, 7, 13, 31, 127])
    q = np.zeros((32, hs.size), dtype=np.uint8)
    for c in range(16):
        for i, v in enumerate(vs):
            q[i] = v + 128
        qw, off, _, _ = O.pack_exl2(q, np.array([8]), np.ones((1, hs.size), np.float16), None)
        codes = np.full((1, hs.size), c, np.uint8)
        pad = (-hs.size) % 8
        codes_p = np.pad(codes, ((0, 0), (0, pad)))
        W = O.dequant_exl2_qscale(np.pad(qw, ((0, 0), (0, pad))), off, np.array([8]), O.pack_exl2_qscale(codes_p),
                                  np.pad(hs, (0, pad)), None)[:, :hs.size]
        mv = O.float64_from_fp16_bits(hs)
        for i, v in enumerate(vs):
            # the rational's value; a zero takes the IEEE sign of the float product
            want = [_py_half_bits(float(Fraction(int(v)) * Fraction(c + 1, 16) * Fraction(float(x))) or
                                  float(v) * float(x)) for x in mv]
            assert np.array_equal(W[i], np.array(want, dtype=np.uint16)), (c, v)


def test_exl2_qscale_packing():
    # nibble i of word k is column 8k + i: columns 0..7 = 1..8 -> 0x87654321
    codes = np.zeros((2, 16), dtype=np.uint8)
    codes[0, :8] = np.arange(1, 9)
    codes[1, 8:] = 15
    w = O.pack_exl2_qscale(codes)
    assert w.tolist() == [[0x87654321, 0], [0, 0xFFFFFFFF]]
    # the same layout as the GPTQ zero points, packed by another function
    rng = np.random.default_rng(3)
    c = rng.integers(0, 16, size=(4, 40)).astype(np.uint8)
    q = np.zeros((4 * 32, 40), dtype=np.uint8)
    _, qz, _, _ = O.pack_gptq(q, c, np.ones((4, 40), np.float16), None, 32)
    assert np.array_equal(O.pack_exl2_qscale(c), qz)
    assert np.array_equal(O.unpack_exl2_qscale(O.pack_exl2_qscale(c), 40), c)
    with pytest.raises(ValueError):
        O.pack_exl2_qscale(np.full((1, 8), 16, np.uint8))


def test_exl2_qscale_dequant_reduces_to_fp16_scales():
    # where ((c + 1) / 16) * m is itself an fp16 value the two-level format is
    # the fp16-scale format with that scale: every code 15 (the scale is the
    # column maximum), and maxima with at most 7 significant bits (any code)
    inp = synth.exl2_layer(256, 48, bpw=4.0, seed=8)
    codes, m = synth.exl2_qscale_draws(8, 48, seed=8)
    qw, off, _, perm = O.pack_exl2(inp.q, inp.bits, inp.s, inp.perm)
    qs = O.pack_exl2_qscale(codes)
    W = O.dequant_exl2_qscale(qw, off, inp.bits, qs, m, perm)
    top = O.pack_exl2_qscale(np.full((8, 48), 15, np.uint8))
    W_top = O.dequant_exl2_qscale(qw, off, inp.bits, top, m, perm)
    assert np.array_equal(W_top, O.dequant_exl2_definitional(inp.q, inp.bits, np.tile(m, (8, 1)), inp.perm))
    m7 = (m.view(np.uint16) & np.uint16(0xFFF0)).view(np.float16)   # 7 significant bits
    s7 = (m7.astype(np.float64)[None, :] * (codes.astype(np.float64) + 1) / 16).astype(np.float16)
    assert np.array_equal(s7.astype(np.float64), m7.astype(np.float64)[None, :] * (codes + 1) / 16)  # exact
    W7 = O.dequant_exl2_qscale(qw, off, inp.bits, qs, m7, perm)
    assert np.array_equal(W7, O.dequant_exl2_definitional(inp.q, inp.bits, s7, inp.perm))
    cols = np.array([0, 9, 47])
    assert np.array_equal(O.dequant_exl2_qscale(qw, off, inp.bits, qs, m, perm, cols=cols), W[:, cols])


# ---------------------------------------------------------------- quantized KV cache codec

def _kv_golden():
    rows = _fixture("kv_codec.txt")
    x = np.array([int(t, 16) for t in rows[0].split()[1:]] + [0] * 24, dtype=np.uint16)
    cases = []
    for row in rows[1:]:
        tok = row.split()
        i_s, i_u, i_w, i_x = tok.index("s"), tok.index("u"), tok.index("words"), tok.index("xhat")
        cases.append((int(tok[1]), int(tok[i_s + 1], 16), [int(t) for t in tok[i_u + 1:i_w]],
                      [int(t, 16) for t in tok[i_w + 1:i_x]], [int(t, 16) for t in tok[i_x + 1:]]))
    return x, cases


def test_kv_codec_golden():
    x, cases = _kv_golden()
    for b, s_want, u_want, words_want, xhat_want in cases:
        u, s = O.kv_quantize(x[None, :], b)
        assert int(s[0]) == s_want, b
        assert u[0, :8].tolist() == u_want, b
        assert (u[0, 8:] == 1 << (b - 1)).all(), b
        words = O.kv_pack(u, b)
        assert [int(w) for w in words[0]] == words_want, b
        assert np.array_equal(O.kv_unpack(words, b, 32), u)
        xh = O.kv_dequantize(words, s, b, 32)
        assert [int(v) for v in xh[0, :8]] == xhat_want, b


def test_kv_codec_properties():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((300, 128)) * np.exp2(rng.integers(-12, 4, (300, 1)))).astype(np.float16)
    x[0] = 0                                    # an all-zero group
    x[1, :] = np.float16(-0.0)
    x[2, 5] = np.float16(65504.0)               # the largest finite value
    x[3, :] = np.float16(2.0 ** -24)            # amax / qmax rounds to a zero scale
    x[4, :] = (rng.standard_normal(128) * 2.0 ** -17).astype(np.float16)  # a subnormal scale at every width
    for b in O.KV_BITS:
        qmax = (1 << (b - 1)) - 1
        u, s = O.kv_quantize(x, b)
        q = u.astype(np.int64) - (1 << (b - 1))
        sv = O.float64_from_fp16_bits(s)
        xv = O.float64_from_fp16_bits(x.view(np.uint16))
        # with a normal fp16 scale (relative rounding <= 2^-11) the amax element
        # takes the largest code; mirrored inputs mirror the codes
        amax_i = np.abs(xv).argmax(axis=1)
        big = sv > 0
        normal = sv >= 2.0 ** -14
        assert normal.sum() > 150 and (~normal & big).any()   # both kinds occur
        assert (np.abs(q[np.arange(300), amax_i])[normal] == qmax).all(), b
        u_neg, s_neg = O.kv_quantize(-x, b)
        q_neg = u_neg.astype(np.int64) - (1 << (b - 1))
        assert np.array_equal(s_neg, s) and np.array_equal(q_neg[normal], -q[normal]), b
        # zero scales give zero codes and +0 outputs
        assert (q[~big] == 0).all() and not big[0] and not big[3], b
        xh = O.float64_from_fp16_bits(O.kv_dequantize(O.kv_pack(u, b), s, b, 128))
        assert (xh[~big] == 0).all() and not np.signbit(xh[~big]).any()
        # |x - xhat| <= s/2 (quotient and code rounding) + half an fp16 ulp of xhat
        err = np.abs(xh - xv)
        bound = 0.5 * sv[:, None] * (1 + 2.0 ** -20) + 0.5 * np.exp2(np.floor(np.log2(np.maximum(np.abs(xh), 2.0 ** -14))) - 10)
        assert (err[normal] <= bound[normal]).all(), b
        # a subnormal scale may clamp the largest codes: the error is then bounded by amax
        assert (err[big & ~normal] <= 2 * np.abs(xv).max(axis=1, keepdims=True)[big & ~normal]).all(), b
        # monotone codes within a group
        order = np.argsort(xv, axis=1, kind="stable")
        assert (np.diff(np.take_along_axis(q, order, axis=1), axis=1) >= 0).all(), b


def test_kv_stream_layout_is_the_exl2_column_stream():
    # a 32-value group packs exactly as one EXL2 segment column of the same width,
    # built by the other packer and by a Python big integer
    rng = np.random.default_rng(4)
    for b in O.KV_BITS:
        u = rng.integers(0, 1 << b, size=(3, 32)).astype(np.uint8)
        words = O.kv_pack(u, b)
        qw, _, _, _ = O.pack_exl2(u.T.copy(), [b], np.ones((1, 3), np.float16), None)
        assert np.array_equal(words, qw.T), b
        stream = sum(int(v) << (i * b) for i, v in enumerate(u[1]))
        assert [int(w) for w in words[1]] == [(stream >> (32 * t)) & 0xFFFFFFFF for t in range(b)], b


def test_kv_codec_ties_round_to_even():
    # s = fp16(1/7) = 1170 x 2^-13; x = 585 x 2^-13 and 1755 x 2^-13 are fp16
    # values whose quotients are exactly 0.5 and 1.5 in fp32: ties go to the
    # even code (0 and 2), also for the negative tie
    x = np.zeros((1, 32), np.float64)
    x[0, :4] = [1.0, 585 * 2.0 ** -13, -585 * 2.0 ** -13, 1755 * 2.0 ** -13]
    u, s = O.kv_quantize(x.astype(np.float16), 4)
    assert int(s[0]) == 0x3092
    assert (u[0, :4].astype(int) - 8).tolist() == [7, 0, 0, 2]


# ---------------------------------------------------------------- EXL2 conversion: RTN, errors, solve

def test_rtn_quantize_matches_the_kv_golden_group():
    # one segment column holding the KV codec's worked group: same scale and codes
    # (two separately written quantizers against the hand-derived fixture)
    x, cases = _kv_golden()
    W = np.zeros((32, 8), dtype=np.uint16)
    W[:, 3] = x
    for b, s_want, u_want, _, _ in cases:
        q, s = O.rtn_quantize_exl2(W, None, [b])
        assert int(s[0, 3]) == s_want, b
        assert q[:8, 3].tolist() == u_want, b


def test_rtn_quantize_roundtrip_and_errors():
    rng = np.random.default_rng(21)
    K, N = 32 * 6, 40
    W = (rng.standard_normal((K, N)) * 0.02).astype(np.float16)
    W[:32] *= 8                                   # one loud segment
    perm = rng.permutation(K).astype(np.int32)
    err = O.rtn_errors_exl2(W, perm)
    Wv = O.float64_from_fp16_bits(W.view(np.uint16))
    for i, b in enumerate(O.EXL2_BITS):
        bits = np.full(K // 32, b)
        q, s = O.rtn_quantize_exl2(W, perm, bits)
        qw, off, sc, pm = O.pack_exl2(q, bits, s.view(np.float16), perm)
        W_hat = O.float64_from_fp16_bits(O.dequant_exl2(qw, off, bits, sc, pm))
        # the error table is the squared error of the whole pipeline, per stored segment
        d2 = ((Wv - W_hat) ** 2)[perm].reshape(K // 32, 32, N).sum(axis=(1, 2))
        assert np.allclose(err[:, i], d2, rtol=1e-12, atol=0), b
        # within half a scale step plus half an fp16 ulp of the result
        sv = O.float64_from_fp16_bits(s)[np.arange(K) // 32][np.argsort(perm)]
        bound = 0.5 * sv + 0.5 * np.exp2(np.floor(np.log2(np.maximum(np.abs(W_hat), 2.0 ** -14))) - 10)
        assert (np.abs(Wv - W_hat) <= bound * (1 + 2.0 ** -20)).all(), b
    assert (np.diff(err, axis=1) <= 0).all()        # more bits, less error (on these weights)


def test_solve_exl2_bits_hand_worked():
    # start 2/2/2 (6 bits); gains per added bit:
    #   seg2 300 -> 3 bits; seg2 70 -> 4; seg0 50 -> 3; seg0 30 -> 4; seg2 20 -> 5;
    #   seg0 10 and seg1 10 tie -> seg0 -> 5 (12 bits); then seg1 10 -> 3 (13 bits)
    err = [[100, 50, 20, 10, 5, 1], [80, 70, 60, 50, 40, 30], [400, 100, 30, 10, 5, 2]]
    assert O.solve_exl2_bits(err, 6).tolist() == [2, 2, 2]
    assert O.solve_exl2_bits(err, 8).tolist() == [2, 2, 4]
    assert O.solve_exl2_bits(err, 12).tolist() == [5, 2, 5]
    assert O.solve_exl2_bits(err, 13).tolist() == [5, 3, 5]
    # the 6 -> 8 step costs two bits: taken when they fit, not when one is left
    one = [[10, 9, 8, 7, 6, 0]]
    assert O.solve_exl2_bits(one, 8).tolist() == [8]
    assert O.solve_exl2_bits(one, 7).tolist() == [6]
    with pytest.raises(ValueError):
        O.solve_exl2_bits(err, 5)


def test_solve_exl2_bits_on_measured_errors():
    rng = np.random.default_rng(5)
    K, N = 32 * 16, 64
    W = (rng.standard_normal((K, N)) * 0.02).astype(np.float16)
    W[64:96] *= 16                                 # segment 2 is far louder
    err = O.rtn_errors_exl2(W, None)
    bits = O.solve_exl2_bits(err, 4 * 16)
    assert int(bits.astype(int).sum()) == 64 and set(bits.tolist()) <= set(O.EXL2_BITS)
    assert bits[2] == bits.max() and bits[2] > 4


def test_exl2_segment_word_offsets_closed_form():
    # a segment of width b packs 32 codes of b bits = b words, so segment s
    # starts at the sum of the widths before it (worked by hand)
    off = O.exl2_seg_word_off([2, 3, 8, 4, 5, 6])
    assert off.dtype == np.uint32
    assert off.tolist() == [0, 2, 5, 13, 17, 22, 28]
    # and it agrees with the packer's own table on a drawn layer
    rng = np.random.default_rng(5)
    bits = rng.choice(O.EXL2_BITS, size=6)
    K, N = 32 * bits.size, 16
    q = np.stack([rng.integers(0, 1 << int(b), size=(32, N)) for b in bits]).reshape(K, N).astype(np.uint8)
    s = np.full((bits.size, N), 0.01, dtype=np.float16)
    qw, off_p = O.pack_exl2(q, bits, s, None)[:2]
    assert np.array_equal(off_p, O.exl2_seg_word_off(bits))
    assert qw.shape == (int(bits.sum()), N)
