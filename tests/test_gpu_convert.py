"""GPU parity of the EXL2 conversion path (RTN quantiser, error table, and the
chain measure -> solve -> quantise -> matmul) against the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
import synth
from helpers import check_matmul

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_exq_gb300 as exq
    torch.cuda.set_device(0)
    return exq, torch


def _weight(K, N, seed):
    """Seeded fp16 weights: N(0, 0.02) per column times a per-row power of two
    in 2^-2 .. 2^2 (rows of different loudness, so that the widths differ)."""
    rng = synth.rng_for(seed, synth.WORKLOAD_IDS["test"], K, N)
    return (rng.standard_normal((K, N)) * 0.02 * np.exp2(rng.integers(-2, 3, (K, 1)))).astype(np.float16)


@pytest.mark.parametrize("K,N,perm", [(32 * 6, 72, True), (1024, 264, False), (2048, 520, True)])
def test_quantize_exl2_bit_exact(env, K, N, perm):
    exq, torch = env
    W = _weight(K, N, seed=K + N)
    S = K // 32
    bits = np.array([2, 3, 4, 5, 6, 8] * (S // 6 + 1))[:S] if S >= 6 else np.full(S, 4)
    p = np.random.default_rng(K).permutation(K).astype(np.int32) if perm else None
    pd = None if p is None else torch.from_numpy(p).cuda()
    w = exq.exq_quantize_exl2(torch.from_numpy(W).cuda(), bits, pd)
    torch.cuda.synchronize()
    assert exq.exq_get_last_device_error() == 0
    q, s = O.rtn_quantize_exl2(W, p, bits)
    oqw, ooff, osc, _ = O.pack_exl2(q, bits, s.view(np.float16), p)
    assert np.array_equal(w.qweight.cpu().numpy().view(np.uint32), oqw)
    assert np.array_equal(w.scales.cpu().numpy().view(np.uint16), osc)
    assert np.array_equal(w.seg_word_off.cpu().numpy().view(np.uint32), ooff)


@pytest.mark.parametrize("K,N,perm", [(32 * 4, 64, False), (1024, 600, True)])
def test_measure_exl2_matches_oracle(env, K, N, perm):
    exq, torch = env
    W = _weight(K, N, seed=3 * K + N)
    p = np.random.default_rng(N).permutation(K).astype(np.int32) if perm else None
    err = exq.exq_measure_exl2(torch.from_numpy(W).cuda(), None if p is None else torch.from_numpy(p).cuda())
    torch.cuda.synchronize()
    ref = O.rtn_errors_exl2(W, p)
    got = err.cpu().numpy().astype(np.float64)
    assert np.allclose(got, ref, rtol=2e-5, atol=0), np.abs(got / ref - 1).max()
    # deterministic
    err2 = exq.exq_measure_exl2(torch.from_numpy(W).cuda(), None if p is None else torch.from_numpy(p).cuda())
    assert torch.equal(err, err2)


def test_convert_chain_then_gemv(env):
    # measure on the GPU, solve on the host for 4.0 bpw, quantise on the GPU,
    # multiply with exq_gemv: against the oracle doing the same from its own table
    exq, torch = env
    K, N = 2048, 264
    p = np.random.default_rng(77).permutation(K).astype(np.int32)
    # loudness per stored segment (its 32 input rows p[32 s: 32 s + 32]), so that the widths differ
    W = _weight(K, N, seed=77).astype(np.float32)
    loud = np.exp2(np.random.default_rng(78).integers(-3, 4, K // 32))
    W[p] *= np.repeat(loud, 32)[:, None]
    W = W.astype(np.float16)
    Wd, pd = torch.from_numpy(W).cuda(), torch.from_numpy(p).cuda()
    ref_err = O.rtn_errors_exl2(W, p)
    bits = exq.exq_solve_exl2_bits(ref_err, 4 * (K // 32))
    assert np.array_equal(bits, O.solve_exl2_bits(ref_err, 4 * (K // 32)))
    assert len(set(bits.tolist())) > 1 and int(bits.astype(int).sum()) == 4 * (K // 32)
    gpu_bits = exq.exq_solve_exl2_bits(exq.exq_measure_exl2(Wd, pd).cpu().numpy().astype(np.float64), 4 * (K // 32))
    assert int(gpu_bits.astype(int).sum()) == int(bits.astype(int).sum())
    w = exq.exq_quantize_exl2(Wd, bits, pd)
    q, s = O.rtn_quantize_exl2(W, p, bits)
    oqw, ooff, osc, op = O.pack_exl2(q, bits, s.view(np.float16), p)
    W_ref = O.dequant_exl2(oqw, ooff, bits, osc, op)
    for M in (1, 8):
        x = synth.activations(M, K, seed=M)
        y = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        exq.exq_gemv(w, torch.from_numpy(x).cuda(), y)
        torch.cuda.synchronize()
        assert exq.exq_get_last_device_error() == 0
        check_matmul(y.float().cpu().numpy().astype(np.float64), O.matmul(x, W_ref), f"converted M={M}")
