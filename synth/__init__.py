"""Seeded synthetic inputs for the quantized-matmul workloads.

This module only draws random inputs: integer codes, fp16 scales, zero points,
bit-width mixes, permutations and activations. It holds none of the method's
arithmetic (no packing, no dequantisation, no matmul), so the CPU oracle and
the CUDA path can both consume its output without sharing any code.

Every array comes from ``numpy.random.default_rng(SeedSequence([seed,
workload, layer, tensor]))``, so each tensor of each layer of each workload is
reproducible on its own. Floating-point draws are made in float32 and rounded
to the fp16 grid (numpy's round-to-nearest-even cast), so scales and
activations are exact fp16 values.

Distributions follow the workloads the ExLlamaV2 pages benchmark (Llama-2-7B
and Llama-2-70B layer shapes; GPTQ 4-bit with 128-row groups; EXL2 at a target
average bits per weight with bit widths 2/3/4/5/6/8):

* GPTQ: q ~ U{0..15}, zero z ~ U{0..15}, scale s ~ U(0.005, 0.02) per
  (group, column); act-order ``g_idx = permutation(K) // group_size``.
* EXL2: 32-row segments; per-segment bit width drawn from a tilted
  distribution whose mean is the target bpw, then nudged by +-1 steps so the
  total number of bits is exactly ``bpw * S``; q ~ U{0..2^b-1}; scale
  s ~ U(0.002, 0.03) per (segment, column); a random permutation of the K
  input features.
* EXL2 with two-level scales: a 4-bit group-scale code c ~ U{0..15} per
  (segment, column) and a column maximum m ~ U(0.02, 0.05) in fp16.
* x ~ N(0, 1) in fp16.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# Tensor ids inside one layer's seed sequence.
_T_Q, _T_Z, _T_S, _T_GIDX, _T_BITS, _T_PERM, _T_X, _T_QSC, _T_SMAX = range(9)

# Workload ids, so that different workloads draw independent streams.
WORKLOAD_IDS = {
    "gptq_gemv_4096": 0,
    "gptq_act_order_7b": 1,
    "exl2_4p0_7b": 2,
    "prefill_70b": 3,
    "decode_stream_70b": 4,
    "test": 99,
}

LLAMA2_7B_SHAPES = {
    # name: (K = in_features, N = out_features)
    "q": (4096, 4096),
    "k": (4096, 4096),
    "v": (4096, 4096),
    "o": (4096, 4096),
    "gate": (4096, 11008),
    "up": (4096, 11008),
    "down": (11008, 4096),
}

LLAMA2_70B_SHAPES = {
    "q": (8192, 8192),
    "k": (8192, 1024),
    "v": (8192, 1024),
    "o": (8192, 8192),
    "gate": (8192, 28672),
    "up": (8192, 28672),
    "down": (28672, 8192),
}

EXL2_BITS = (2, 3, 4, 5, 6, 8)
SEGMENT_ROWS = 32


def rng_for(seed: int, workload: int, layer: int, tensor: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, workload, layer, tensor]))


def fp16_uniform(rng: np.random.Generator, lo: float, hi: float, shape) -> np.ndarray:
    return rng.uniform(lo, hi, size=shape).astype(np.float32).astype(np.float16)


def activations(M: int, K: int, seed: int = 0, workload: int = 99, layer: int = 0) -> np.ndarray:
    """x ~ N(0,1), fp16 [M, K] row-major."""
    rng = rng_for(seed, workload, layer, _T_X)
    return rng.standard_normal(size=(M, K), dtype=np.float32).astype(np.float16)


@dataclass
class GptqInputs:
    """Unpacked GPTQ layer, rows in ORIGINAL input-feature order."""

    q: np.ndarray       # uint8 [K, N], 0..15
    z: np.ndarray       # uint8 [G, N], 0..15
    s: np.ndarray       # float16 [G, N]
    g_idx: np.ndarray   # int32 [K], group of original row k
    group_size: int

    @property
    def K(self) -> int:
        return self.q.shape[0]

    @property
    def N(self) -> int:
        return self.q.shape[1]


def gptq_layer(K: int, N: int, group_size: int = 128, act_order: bool = False,
               seed: int = 0, workload: int = 99, layer: int = 0,
               s_range=(0.005, 0.02)) -> GptqInputs:
    if K % group_size:
        raise ValueError("K must be a multiple of group_size")
    G = K // group_size
    q = rng_for(seed, workload, layer, _T_Q).integers(0, 16, size=(K, N), dtype=np.uint8)
    z = rng_for(seed, workload, layer, _T_Z).integers(0, 16, size=(G, N), dtype=np.uint8)
    s = fp16_uniform(rng_for(seed, workload, layer, _T_S), s_range[0], s_range[1], (G, N))
    if act_order:
        g_idx = (rng_for(seed, workload, layer, _T_GIDX).permutation(K) // group_size)
    else:
        g_idx = np.arange(K) // group_size
    return GptqInputs(q=q, z=z, s=s, g_idx=g_idx.astype(np.int32), group_size=group_size)


def solve_bit_mix(S: int, bpw: float, allowed=EXL2_BITS, rng: np.random.Generator | None = None,
                  step_range=None) -> np.ndarray:
    """Draw S per-segment bit widths from ``allowed`` whose sum is exactly bpw*S.

    Seeded preference weights w_b are tilted to p_b ~ w_b * exp(lam*b) with lam
    found by bisection so that E[b] = bpw; S widths are drawn i.i.d.; then
    random +-1 steps (only between widths inside ``step_range``, default
    2..6) fix the total exactly. This stands in for the EXL2 converter's solve
    pass, which needs calibration data.
    """
    if rng is None:
        rng = np.random.default_rng(0)
    allowed = np.array(sorted(allowed), dtype=np.int64)
    target = bpw * S
    if abs(target - round(target)) > 1e-9:
        raise ValueError("bpw * S must be an integer")
    target = int(round(target))
    if not (allowed.min() * S <= target <= allowed.max() * S):
        raise ValueError("bpw outside the allowed bit widths")
    w = rng.uniform(0.5, 1.5, size=allowed.size)

    def mean(lam):
        p = w * np.exp(lam * (allowed - allowed.mean()))
        p /= p.sum()
        return float((p * allowed).sum()), p

    lo, hi = -50.0, 50.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if mean(mid)[0] < bpw:
            lo = mid
        else:
            hi = mid
    _, p = mean(0.5 * (lo + hi))
    bits = rng.choice(allowed, size=S, p=p)
    if step_range is None:
        step_range = (int(allowed.min()), min(6, int(allowed.max())))
    a, b = step_range
    total = int(bits.sum())
    while total != target:
        if total < target:
            cand = np.flatnonzero((bits >= a) & (bits < b))
            j = cand[rng.integers(0, cand.size)]
            bits[j] += 1
            total += 1
        else:
            cand = np.flatnonzero((bits > a) & (bits <= b))
            j = cand[rng.integers(0, cand.size)]
            bits[j] -= 1
            total -= 1
    assert set(np.unique(bits)).issubset(set(allowed.tolist()) | set(range(a, b + 1)))
    return bits.astype(np.uint8)


@dataclass
class Exl2Inputs:
    """Unpacked EXL2 layer, rows in STORED order (stored row j = original row perm[j])."""

    q: np.ndarray      # uint8 [K, N]; row j uses bits[j // 32]
    bits: np.ndarray   # uint8 [S]
    s: np.ndarray      # float16 [S, N]
    perm: np.ndarray   # int32 [K] or None (identity)

    @property
    def K(self) -> int:
        return self.q.shape[0]

    @property
    def N(self) -> int:
        return self.q.shape[1]


def exl2_layer(K: int, N: int, bpw: float = 4.0, allowed=EXL2_BITS, permute: bool = True,
               seed: int = 0, workload: int = 99, layer: int = 0,
               s_range=(0.002, 0.03), bits: np.ndarray | None = None) -> Exl2Inputs:
    if K % SEGMENT_ROWS:
        raise ValueError("K must be a multiple of 32")
    S = K // SEGMENT_ROWS
    if bits is None:
        bits = solve_bit_mix(S, bpw, allowed, rng_for(seed, workload, layer, _T_BITS))
    bits = np.asarray(bits, dtype=np.uint8)
    rng_q = rng_for(seed, workload, layer, _T_Q)
    q = np.empty((K, N), dtype=np.uint8)
    for b in np.unique(bits):
        rows = np.flatnonzero(np.repeat(bits, SEGMENT_ROWS) == b)
        q[rows] = rng_q.integers(0, 1 << int(b), size=(rows.size, N), dtype=np.uint16).astype(np.uint8)
    s = fp16_uniform(rng_for(seed, workload, layer, _T_S), s_range[0], s_range[1], (S, N))
    perm = rng_for(seed, workload, layer, _T_PERM).permutation(K).astype(np.int32) if permute else None
    return Exl2Inputs(q=q, bits=bits, s=s, perm=perm)


def exl2_qscale_draws(S: int, N: int, seed: int = 0, workload: int = 99, layer: int = 0,
                      m_range=(0.02, 0.05)):
    """Two-level EXL2 scale inputs: codes uint8 [S, N] ~ U{0..15} and column
    maxima fp16 [N] ~ U(m_range)."""
    codes = rng_for(seed, workload, layer, _T_QSC).integers(0, 16, size=(S, N)).astype(np.uint8)
    m = fp16_uniform(rng_for(seed, workload, layer, _T_SMAX), m_range[0], m_range[1], (N,))
    return codes, m


def uniform_words(n_words: int, seed: int = 0, workload: int = 4, layer: int = 0) -> np.ndarray:
    """Uniform random uint32 words (a packed stream of uniform codes, by the
    packing bijection: b words per 32-row segment column <-> 32 b-bit codes)."""
    return rng_for(seed, workload, layer, _T_Q).integers(0, 1 << 32, size=n_words, dtype=np.uint64).astype(np.uint32)
