"""GPU parity of exq_gemm_multi (several prefill matmuls that read the same x
in one launch) against the CPU oracle, through the C ABI: every output y_i
within max(2e-2, 1 fp16 ulp) element-wise and rel-L2 <= 1e-3 per row of
x . W_i, NaN-poisoned outputs fully overwritten."""
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


def _exl2_dev(exq, e):
    qw, off = exq.exq_pack_exl2(e.q, e.bits)
    return exq.exl2_weight(qw, off, e.s, e.perm, e.K, e.N)


def _gptq_dev(exq, g):
    qw, qz, perm = exq.exq_pack_gptq(g.q, g.z, g.g_idx, g.group_size)
    has_perm = not np.array_equal(perm, np.arange(g.K))
    return exq.gptq_weight(qw, qz, g.s, perm if has_perm else None, g.K, g.N, g.group_size)


def _multi(exq, torch, ws, x16):
    M = x16.shape[0]
    x = torch.from_numpy(np.ascontiguousarray(x16)).cuda()
    ys = [torch.full((M, w.N), float("nan"), dtype=torch.float16, device="cuda") for w in ws]
    exq.exq_gemm_multi(ws, x, ys)
    torch.cuda.synchronize()
    assert exq.exq_get_last_device_error() == 0
    return [y.float().cpu().numpy().astype(np.float64) for y in ys]


@pytest.mark.parametrize("M", [1, 77, 300])
def test_gemm_multi_exl2_mixed_perms(env, M):
    exq, torch = env
    K = 1024
    # three layers of one K: two with their own permutations, one in input order
    es = [exl2_case(K, 256, bpw=4.0, seed=31), exl2_case(K, 128, bpw=2.5, allowed=(2, 3, 4), seed=32),
          exl2_case(K, 384, bpw=4.0, permute=False, seed=33)]
    x = synth.activations(M, K, seed=M + 30)
    ys = _multi(exq, torch, [_exl2_dev(exq, e) for e in es], x)
    for i, (e, y) in enumerate(zip(es, ys)):
        check_matmul(y, O.matmul(x, oracle_W_exl2(e)), f"multi exl2 layer {i} M={M}")


@pytest.mark.parametrize("M", [64, 256])
def test_gemm_multi_gptq(env, M):
    exq, torch = env
    K = 512
    gs = [gptq_case(K, 256, 128, act_order=True, seed=41), gptq_case(K, 128, 128, act_order=False, seed=42)]
    x = synth.activations(M, K, seed=M + 40)
    ys = _multi(exq, torch, [_gptq_dev(exq, g) for g in gs], x)
    for i, (g, y) in enumerate(zip(gs, ys)):
        check_matmul(y, O.matmul(x, oracle_W_gptq(g)), f"multi gptq layer {i} M={M}")


def test_gemm_multi_matches_unsplit_single_calls(env):
    exq, torch = env
    # with enough tiles no single call splits K, so each grouped output has the
    # bits of its own exq_gemm
    K, M = 512, 512
    es = [exl2_case(K, 1024, bpw=4.0, seed=51), exl2_case(K, 640, bpw=4.0, seed=52)]
    ws = [_exl2_dev(exq, e) for e in es]
    x16 = synth.activations(M, K, seed=50)
    ys = _multi(exq, torch, ws, x16)
    x = torch.from_numpy(x16).cuda()
    for w, y in zip(ws, ys):
        y1 = torch.full((M, w.N), float("nan"), dtype=torch.float16, device="cuda")
        nws = exq.exq_gemm_workspace_size(w, M)
        wsb = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
        exq.exq_gemm(w, x, y1, wsb)
        torch.cuda.synchronize()
        assert np.array_equal(y1.float().cpu().numpy().astype(np.float64), y)


def test_gemm_multi_per_layer_launches_match_single_calls(env):
    exq, torch = env
    # q + k + v shaped like a grouped-query block at M = 512: pooled, the 160
    # tiles would take two waves on 152 SMs, so the call launches per layer
    # and splits the small layers along K as exq_gemm does; the permuted
    # layers read their own slice of the once-gathered activations
    K, M = 4096, 512
    es = [exl2_case(K, 8192, bpw=4.0, seed=71), exl2_case(K, 1024, bpw=4.0, permute=False, seed=72),
          exl2_case(K, 1024, bpw=3.0, allowed=(2, 3, 4), seed=73)]
    ws = [_exl2_dev(exq, e) for e in es]
    x16 = synth.activations(M, K, seed=70)
    ys = _multi(exq, torch, ws, x16)
    x = torch.from_numpy(x16).cuda()
    per_layer = torch.cuda.get_device_properties(0).multi_processor_count == 152
    rng = np.random.default_rng(70)
    for i, (e, w, y) in enumerate(zip(es, ws, ys)):
        cols = np.unique(np.concatenate([rng.choice(w.N, 64, replace=False), [0, w.N - 1]]))
        check_matmul(y[:, cols], O.matmul(x16, oracle_W_exl2(e, cols=cols)), f"multi per-layer {i}")
        y1 = torch.full((M, w.N), float("nan"), dtype=torch.float16, device="cuda")
        wsb = torch.empty(max(exq.exq_gemm_workspace_size(w, M), 16), dtype=torch.uint8, device="cuda")
        exq.exq_gemm(w, x, y1, wsb)
        torch.cuda.synchronize()
        if per_layer or i == 0:  # q alone never splits K at M = 512
            assert np.array_equal(y1.float().cpu().numpy().astype(np.float64), y), f"layer {i}"


def test_gemm_multi_qkv_70b(env):
    exq, torch = env
    # the Llama-2-70B q, k, v projections at M = 512, act-order GPTQ, one launch
    wid = synth.WORKLOAD_IDS["prefill_70b"]
    shapes = [synth.LLAMA2_70B_SHAPES[n] for n in ("q", "k", "v")]
    gs = [gptq_case(K, N, 128, act_order=True, seed=0, workload=wid, layer=30 + i) for i, (K, N) in enumerate(shapes)]
    x = synth.activations(512, shapes[0][0], seed=7, workload=wid)
    ys = _multi(exq, torch, [_gptq_dev(exq, g) for g in gs], x)
    rng = np.random.default_rng(5)
    for i, (g, y) in enumerate(zip(gs, ys)):
        cols = np.unique(np.concatenate([rng.choice(g.N, 96, replace=False), [0, g.N - 1]]))
        check_matmul(y[:, cols], O.matmul(x, oracle_W_gptq(g, cols=cols)), f"multi qkv 70b layer {i}")


def test_gemm_multi_rejects_bad_groups(env):
    exq, torch = env
    e = exl2_case(512, 128, seed=61)
    g = gptq_case(512, 128, 128, seed=62)
    we, wg = _exl2_dev(exq, e), _gptq_dev(exq, g)
    x = torch.zeros(8, 512, dtype=torch.float16, device="cuda")
    ys = [torch.zeros(8, 128, dtype=torch.float16, device="cuda") for _ in range(5)]
    with pytest.raises(exq.ExqError) as ei:
        exq.exq_gemm_multi([we, wg], x, ys[:2])  # mixed formats
    assert ei.value.status == exq.EXQ_ERR_INVALID_ARG
    with pytest.raises(exq.ExqError) as ei:
        exq.exq_gemm_multi([we] * 5, x, ys)  # more than EXQ_GEMM_MAX_LAYERS
    assert ei.value.status == exq.EXQ_ERR_INVALID_ARG
    e64 = exl2_case(512, 64, seed=63)  # N % 128 != 0
    with pytest.raises(exq.ExqError) as ei:
        exq.exq_gemm_multi([we, _exl2_dev(exq, e64)], x, [ys[0], torch.zeros(8, 64, dtype=torch.float16,
                                                                            device="cuda")])
    assert ei.value.status == exq.EXQ_ERR_UNSUPPORTED
