"""Shared test helpers: build packed layers from synthetic inputs with both
the library packer and the oracle, and compare matmul outputs."""
from __future__ import annotations

import numpy as np

import oracle as O
import synth


def ulp16(v):
    """Spacing of fp16 values at |v| (subnormal spacing below 2^-14)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return np.exp2(e - 10)


def check_matmul(got, ref, where=""):
    """|y - y_ref| <= max(2e-2, 1 fp16 ulp of y_ref) element-wise and
    ||y - y_ref|| <= 1e-3 ||y_ref|| per output row (over N)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, where
    assert np.isfinite(got).all(), f"{where}: non-finite output (unwritten element?)"
    err = np.abs(got - ref)
    tol = np.maximum(2e-2, ulp16(ref))
    bad = err > tol
    assert not bad.any(), f"{where}: {bad.sum()} elements out of tolerance, max abs err {err.max():.4g}"
    num = np.linalg.norm(got - ref, axis=1)
    den = np.linalg.norm(ref, axis=1)
    rel = np.where(den > 0, num / np.where(den > 0, den, 1), num)
    assert np.all(rel <= 1e-3), f"{where}: per-row rel-L2 {rel.max():.3g}"
    assert np.all(np.where(den == 0, num == 0, True)), f"{where}: zero row not reproduced"
    return float(err.max()), float(rel.max())


def gptq_case(K, N, gs=128, act_order=False, seed=0, workload=99, layer=0):
    g = synth.gptq_layer(K, N, gs, act_order=act_order, seed=seed, workload=workload, layer=layer)
    return g


def exl2_case(K, N, bpw=4.0, allowed=synth.EXL2_BITS, permute=True, seed=0, bits=None, workload=99, layer=0):
    return synth.exl2_layer(K, N, bpw=bpw, allowed=allowed, permute=permute, seed=seed, bits=bits,
                            workload=workload, layer=layer)


def oracle_W_gptq(g, cols=None):
    qw, qz, sc, perm = O.pack_gptq(g.q, g.z, g.s, g.g_idx, g.group_size)
    return O.dequant_gptq(qw, qz, sc, perm, g.K, g.group_size, cols=cols)


def oracle_W_exl2(e, cols=None):
    qw, off, sc, perm = O.pack_exl2(e.q, e.bits, e.s, e.perm)
    return O.dequant_exl2(qw, off, e.bits, sc, perm, cols=cols)
