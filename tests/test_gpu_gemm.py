"""GPU parity of exq_gemm (tcgen05 prefill path) against the CPU oracle,
through the C ABI: max(2e-2, 1 fp16 ulp) element-wise and rel-L2 <= 1e-3 per
output row."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
import synth
from helpers import check_matmul, exl2_case, gptq_case, oracle_W_exl2, oracle_W_gptq

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_exq_gb300 as exq
    torch.cuda.set_device(0)
    return exq, torch


def _gptq_dev(exq, g, force_perm=False):
    qw, qz, perm = exq.exq_pack_gptq(g.q, g.z, g.g_idx, g.group_size)
    has_perm = force_perm or not np.array_equal(perm, np.arange(g.K))
    return exq.gptq_weight(qw, qz, g.s, perm if has_perm else None, g.K, g.N, g.group_size)


def _exl2_dev(exq, e):
    qw, off = exq.exq_pack_exl2(e.q, e.bits)
    return exq.exl2_weight(qw, off, e.s, e.perm, e.K, e.N)


def _gemm(exq, torch, w, x16):
    M = x16.shape[0]
    x = torch.from_numpy(np.ascontiguousarray(x16)).cuda()
    y = torch.full((M, w.N), float("nan"), dtype=torch.float16, device="cuda")
    nws = exq.exq_gemm_workspace_size(w, M)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda") if nws else None
    exq.exq_gemm(w, x, y, ws)
    torch.cuda.synchronize()
    assert exq.exq_get_last_device_error() == 0
    return y.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M", [1, 77, 128, 300])
@pytest.mark.parametrize("K,N,gs,act", [(128, 256, 128, False), (512, 384, 128, True), (256, 512, 32, True),
                                        (1024, 256, 64, False)])
def test_gemm_gptq_small(env, M, K, N, gs, act):
    exq, torch = env
    g = gptq_case(K, N, gs, act_order=act, seed=K + N + M)
    x = synth.activations(M, K, seed=M)
    y = _gemm(exq, torch, _gptq_dev(exq, g), x)
    check_matmul(y, O.matmul(x, oracle_W_gptq(g)), f"gemm gptq K={K} N={N} M={M}")


@pytest.mark.parametrize("M", [5, 128, 257])
@pytest.mark.parametrize("K,N,bits,perm", [
    (192 * 2, 256, np.array([2, 3, 4, 5, 6, 8, 8, 6, 5, 4, 3, 2]), True),
    (1024, 384, 2.5, True), (512, 256, 4.0, False),
])
def test_gemm_exl2_small(env, M, K, N, bits, perm):
    exq, torch = env
    kw = dict(bits=bits) if isinstance(bits, np.ndarray) else dict(bpw=bits, allowed=(2, 3, 4) if bits < 3 else synth.EXL2_BITS)
    e = exl2_case(K, N, permute=perm, seed=K + N + M, **kw)
    x = synth.activations(M, K, seed=M + 7)
    y = _gemm(exq, torch, _exl2_dev(exq, e), x)
    check_matmul(y, O.matmul(x, oracle_W_exl2(e)), f"gemm exl2 K={K} N={N} M={M}")


def test_gemm_one_hot_rows_exact(env):
    exq, torch = env
    g = gptq_case(512, 256, 128, act_order=True, seed=3)
    W = oracle_W_gptq(g)
    ks = np.arange(0, 512, 4)
    x = np.zeros((128, 512), np.float16)
    x[np.arange(128), ks] = 1.0
    y = _gemm(exq, torch, _gptq_dev(exq, g), x)
    assert np.array_equal(y, O.float64_from_fp16_bits(W[ks]))


def test_gemm_deterministic(env):
    exq, torch = env
    e = exl2_case(2048, 512, bpw=4.0, seed=4)
    w = _exl2_dev(exq, e)
    x = synth.activations(256, 2048, seed=4)
    a = _gemm(exq, torch, w, x)
    b = _gemm(exq, torch, w, x)
    assert np.array_equal(a, b)


def test_gemm_unsupported_shapes(env):
    exq, torch = env
    g = gptq_case(192, 64, 32, seed=5)  # N = 64 is not a multiple of 128
    w = _gptq_dev(exq, g)
    x = torch.zeros(4, 192, dtype=torch.float16, device="cuda")
    y = torch.zeros(4, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(exq.ExqError) as ei:
        exq.exq_gemm(w, x, y)
    assert ei.value.status == exq.EXQ_ERR_UNSUPPORTED


def _sample_cols(N, n=192, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.choice(N, n, replace=False), [0, N - 1]]))


@pytest.mark.parametrize("name", ["k", "q", "down"])
def test_prefill_70b_gptq(env, name):
    exq, torch = env
    K, N = synth.LLAMA2_70B_SHAPES[name]
    wid = synth.WORKLOAD_IDS["prefill_70b"]
    g = gptq_case(K, N, 128, act_order=False, seed=0, workload=wid, layer=list(synth.LLAMA2_70B_SHAPES).index(name))
    w = _gptq_dev(exq, g)
    cols = _sample_cols(N, seed=K)
    W_ref = oracle_W_gptq(g, cols=cols)
    x = synth.activations(512, K, seed=1, workload=wid)
    check_matmul(_gemm(exq, torch, w, x)[:, cols], O.matmul(x, W_ref), f"prefill gptq {name}")


@pytest.mark.parametrize("name", ["v", "up"])
def test_prefill_70b_exl2_2p5(env, name):
    exq, torch = env
    K, N = synth.LLAMA2_70B_SHAPES[name]
    wid = synth.WORKLOAD_IDS["prefill_70b"]
    e = exl2_case(K, N, bpw=2.5, allowed=(2, 3, 4), seed=0, workload=wid,
                  layer=10 + list(synth.LLAMA2_70B_SHAPES).index(name))
    w = _exl2_dev(exq, e)
    cols = _sample_cols(N, seed=K + 3)
    W_ref = oracle_W_exl2(e, cols=cols)
    x = synth.activations(512, K, seed=2, workload=wid)
    check_matmul(_gemm(exq, torch, w, x)[:, cols], O.matmul(x, W_ref), f"prefill exl2 {name}")


# The prefill sizes the benchmark quotes: the 70B gate shape at M = 2048, and
# the permuted variants (x gathered pair-interleaved, the XP kernels) at 70B
# sizes; sampled columns against the oracle, y poisoned with NaN.

def test_prefill_70b_gate_m2048_gptq(env):
    exq, torch = env
    K, N = synth.LLAMA2_70B_SHAPES["gate"]
    wid = synth.WORKLOAD_IDS["prefill_70b"]
    g = gptq_case(K, N, 128, act_order=False, seed=0, workload=wid, layer=4)
    cols = _sample_cols(N, n=128, seed=K + 11)
    x = synth.activations(2048, K, seed=3, workload=wid)
    y = _gemm(exq, torch, _gptq_dev(exq, g), x)
    check_matmul(y[:, cols], O.matmul(x, oracle_W_gptq(g, cols=cols)), "prefill gptq gate M=2048")


def test_prefill_70b_gate_m2048_exl2_2p5(env):
    exq, torch = env
    K, N = synth.LLAMA2_70B_SHAPES["gate"]
    wid = synth.WORKLOAD_IDS["prefill_70b"]
    e = exl2_case(K, N, bpw=2.5, allowed=(2, 3, 4), permute=False, seed=0, workload=wid, layer=14)
    cols = _sample_cols(N, n=128, seed=K + 12)
    x = synth.activations(2048, K, seed=4, workload=wid)
    y = _gemm(exq, torch, _exl2_dev(exq, e), x)
    check_matmul(y[:, cols], O.matmul(x, oracle_W_exl2(e, cols=cols)), "prefill exl2 2.5 gate M=2048")


def test_prefill_70b_q_act_order_gptq(env):
    exq, torch = env
    K, N = synth.LLAMA2_70B_SHAPES["q"]
    wid = synth.WORKLOAD_IDS["prefill_70b"]
    g = gptq_case(K, N, 128, act_order=True, seed=0, workload=wid, layer=20)
    w = _gptq_dev(exq, g)
    assert w.perm is not None
    cols = _sample_cols(N, n=128, seed=K + 13)
    x = synth.activations(512, K, seed=5, workload=wid)
    check_matmul(_gemm(exq, torch, w, x)[:, cols], O.matmul(x, oracle_W_gptq(g, cols=cols)),
                 "prefill gptq act-order q")


def test_prefill_70b_down_permuted_exl2_2p5(env):
    exq, torch = env
    K, N = synth.LLAMA2_70B_SHAPES["down"]
    wid = synth.WORKLOAD_IDS["prefill_70b"]
    e = exl2_case(K, N, bpw=2.5, allowed=(2, 3, 4), permute=True, seed=0, workload=wid, layer=21)
    w = _exl2_dev(exq, e)
    assert w.perm is not None
    cols = _sample_cols(N, n=128, seed=K + 14)
    x = synth.activations(512, K, seed=6, workload=wid)
    check_matmul(_gemm(exq, torch, w, x)[:, cols], O.matmul(x, oracle_W_exl2(e, cols=cols)),
                 "prefill exl2 2.5 permuted down")
