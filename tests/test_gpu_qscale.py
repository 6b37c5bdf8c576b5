"""GPU parity of the EXL2 two-level-scale format (4-bit group-scale codes x
per-column fp16 maxima) against the CPU oracle, through the C ABI, on every
device op: dequant bit-exact; decode GEMV, grouped GEMV and prefill GEMM
within max(2e-2, 1 fp16 ulp) element-wise and rel-L2 <= 1e-3 per output row."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
import synth
from helpers import check_matmul, exl2_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_exq_gb300 as exq
    torch.cuda.set_device(0)
    return exq, torch


def _case(exq, K, N, bpw=4.0, bits=None, permute=True, seed=0, workload=99, layer=0):
    """(device layer, oracle W [K, N] fp16 bits, oracle inputs)."""
    kw = dict(bits=bits) if bits is not None else dict(bpw=bpw, allowed=(2, 3, 4) if bpw < 3 else synth.EXL2_BITS)
    e = exl2_case(K, N, permute=permute, seed=seed, workload=workload, layer=layer, **kw)
    codes, m = synth.exl2_qscale_draws(K // 32, N, seed=seed, workload=workload, layer=layer)
    qw, off = exq.exq_pack_exl2(e.q, e.bits)
    w = exq.exl2_qscale_weight(qw, off, exq.exq_pack_exl2_qscale(codes), m, e.perm, K, N)
    oqw, ooff, _, operm = O.pack_exl2(e.q, e.bits, e.s, e.perm)
    return w, (oqw, ooff, e.bits, O.pack_exl2_qscale(codes), m.view(np.uint16), operm)


def _oracle_W(ref, cols=None):
    oqw, ooff, bits, oqs, m, operm = ref
    return O.dequant_exl2_qscale(oqw, ooff, bits, oqs, m, operm, cols=cols)


def _x(torch, x16):
    return torch.from_numpy(np.ascontiguousarray(x16)).cuda()


def _dequant(exq, torch, w):
    W = torch.full((w.K, w.N), float("nan"), dtype=torch.float16, device="cuda")
    exq.exq_dequant(w, W)
    torch.cuda.synchronize()
    assert exq.exq_get_last_device_error() == 0
    return W.cpu().numpy().view(np.uint16)


def _gemv(exq, torch, w, x16, workspace=None):
    y = torch.full((x16.shape[0], w.N), float("nan"), dtype=torch.float16, device="cuda")
    exq.exq_gemv(w, _x(torch, x16), y, workspace=workspace)
    torch.cuda.synchronize()
    assert exq.exq_get_last_device_error() == 0
    return y.float().cpu().numpy().astype(np.float64)


def _gemm(exq, torch, w, x16):
    M = x16.shape[0]
    y = torch.full((M, w.N), float("nan"), dtype=torch.float16, device="cuda")
    nws = exq.exq_gemm_workspace_size(w, M)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda") if nws else None
    exq.exq_gemm(w, _x(torch, x16), y, ws)
    torch.cuda.synchronize()
    assert exq.exq_get_last_device_error() == 0
    return y.float().cpu().numpy().astype(np.float64)


SMALL = [  # K, N, bits / bpw, permute
    (1024, 200, 4.0, True), (32 * 6, 72, np.array([2, 3, 4, 5, 6, 8]), True),
    (32 * 12, 64, np.array([8, 8, 6, 6, 5, 5, 3, 3, 2, 2, 4, 4]), False), (2048, 264, 2.5, True),
]


def _small(exq, K, N, bits, perm, seed):
    if isinstance(bits, np.ndarray):
        return _case(exq, K, N, bits=bits, permute=perm, seed=seed)
    return _case(exq, K, N, bpw=bits, permute=perm, seed=seed)


@pytest.mark.parametrize("K,N,bits,perm", SMALL)
def test_qscale_dequant_bit_exact(env, K, N, bits, perm):
    exq, torch = env
    w, ref = _small(exq, K, N, bits, perm, seed=K + N)
    assert np.array_equal(_dequant(exq, torch, w), _oracle_W(ref))


def test_qscale_dequant_special_maxima(env):
    # subnormal, negative, zero and the largest finite maxima; every code
    exq, torch = env
    K, N = 256, 64
    e = exl2_case(K, N, bits=np.array([4] * 8), permute=False, seed=1)
    codes = np.tile(np.arange(16, dtype=np.uint8), (8, 4))
    m = np.zeros(N, np.float16)
    m[:16] = np.float16(2.0 ** -20)
    m[16:32] = np.float16(-0.7)
    m[32:40] = np.float16(0.0)
    m[40:48] = np.float16(65504.0)
    m[48:] = np.float16(3.0 * 2.0 ** -24)
    qw, off = exq.exq_pack_exl2(e.q, e.bits)
    w = exq.exl2_qscale_weight(qw, off, exq.exq_pack_exl2_qscale(codes), m, None, K, N)
    oqw, ooff, _, _ = O.pack_exl2(e.q, e.bits, e.s, None)
    W_ref = O.dequant_exl2_qscale(oqw, ooff, e.bits, O.pack_exl2_qscale(codes), m.view(np.uint16), None)
    assert np.array_equal(_dequant(exq, torch, w), W_ref)


@pytest.mark.parametrize("M", [1, 5, 16])
@pytest.mark.parametrize("K,N,bits,perm", SMALL)
def test_qscale_gemv_small(env, M, K, N, bits, perm):
    exq, torch = env
    w, ref = _small(exq, K, N, bits, perm, seed=K + N)
    x = synth.activations(M, K, seed=M + 30)
    check_matmul(_gemv(exq, torch, w, x), O.matmul(x, _oracle_W(ref)), f"qscale gemv K={K} N={N} M={M}")


@pytest.mark.parametrize("ctas", [1, 37, 1000])
def test_qscale_gemv_any_split(env, ctas, monkeypatch):
    exq, torch = env
    monkeypatch.setenv("EXQ_GEMV_CTAS", str(ctas))
    w, ref = _case(exq, 2048, 200, seed=ctas)
    for M in (1, 9):
        x = synth.activations(M, 2048, seed=M + ctas)
        ws = torch.zeros(exq.exq_gemv_workspace_size(w, M), dtype=torch.uint8, device="cuda")
        check_matmul(_gemv(exq, torch, w, x, workspace=ws), O.matmul(x, _oracle_W(ref)), f"ctas={ctas} M={M}")
        assert int(ws[:65536].view(torch.int32).abs().sum()) == 0


def test_qscale_gemv_multi(env):
    exq, torch = env
    layers = [_case(exq, 1024, N, seed=40 + i, permute=p) for i, (N, p) in enumerate(((256, True), (64, False),
                                                                                      (136, True)))]
    for M in (1, 12):
        x = synth.activations(M, 1024, seed=M)
        ys = [torch.full((M, w.N), float("nan"), dtype=torch.float16, device="cuda") for w, _ in layers]
        exq.exq_gemv_multi([w for w, _ in layers], _x(torch, x), ys)
        torch.cuda.synchronize()
        assert exq.exq_get_last_device_error() == 0
        for i, (y, (_, ref)) in enumerate(zip(ys, layers)):
            check_matmul(y.float().cpu().numpy().astype(np.float64), O.matmul(x, _oracle_W(ref)),
                         f"qscale group layer {i} M={M}")


@pytest.mark.parametrize("M", [5, 128, 300])
@pytest.mark.parametrize("K,N,bits,perm", [
    (192 * 2, 256, np.array([2, 3, 4, 5, 6, 8, 8, 6, 5, 4, 3, 2]), True), (1024, 384, 2.5, True),
    (512, 128, 4.0, False),
])
def test_qscale_gemm(env, M, K, N, bits, perm):
    exq, torch = env
    w, ref = _small(exq, K, N, bits, perm, seed=K + N + M)
    x = synth.activations(M, K, seed=M + 9)
    check_matmul(_gemm(exq, torch, w, x), O.matmul(x, _oracle_W(ref)), f"qscale gemm K={K} N={N} M={M}")


def _sample_cols(N, n=160, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.choice(N, n, replace=False), [0, N - 1]]))


def test_qscale_70b_gate_sampled(env):
    # the 70B gate shape at 4.0 bpw: decode (M = 1) and prefill (M = 512), sampled columns
    exq, torch = env
    K, N = synth.LLAMA2_70B_SHAPES["gate"]
    w, ref = _case(exq, K, N, seed=0, workload=synth.WORKLOAD_IDS["decode_stream_70b"], layer=4)
    cols = _sample_cols(N, seed=5)
    W_ref = _oracle_W(ref, cols=cols)
    assert np.array_equal(_dequant(exq, torch, w)[:, cols], W_ref)
    x1 = synth.activations(1, K, seed=1)
    check_matmul(_gemv(exq, torch, w, x1)[:, cols], O.matmul(x1, W_ref), "qscale 70b gate gemv")
    x512 = synth.activations(512, K, seed=2)
    check_matmul(_gemm(exq, torch, w, x512)[:, cols], O.matmul(x512, W_ref), "qscale 70b gate gemm")
