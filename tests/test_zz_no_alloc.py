"""exq_gemm_noalloc: the prefill matmul for callers that cannot allocate
device memory (for example an inference-runtime plugin whose enqueue path
must not allocate, or a serving loop that cannot afford cudaMalloc's implicit
device synchronisation). It must give the same results as exq_gemm with a
caller-provided workspace, call after call, while the library's static
scratch array is reused.

This file is named so that pytest collects it last."""
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


def _layer(exq, K, N, seed):
    g = gptq_case(K, N, 128, act_order=True, seed=seed)
    qw, qz, perm = exq.exq_pack_gptq(g.q, g.z, g.g_idx, g.group_size)
    return g, exq.gptq_weight(qw, qz, g.s, perm, g.K, g.N, g.group_size)


def _with_workspace(exq, torch, w, x):
    y = torch.full((x.shape[0], w.N), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.empty(exq.exq_gemm_workspace_size(w, x.shape[0]), dtype=torch.uint8, device="cuda")
    exq.exq_gemm(w, x, y, ws)
    return y


def _without(exq, torch, w, x):
    y = torch.full((x.shape[0], w.N), float("nan"), dtype=torch.float16, device="cuda")
    exq.exq_gemm_noalloc(w, x, y)
    return y


def test_noalloc_matches_workspace_path_two_calls(env):
    exq, torch = env
    # two different act-order layers and inputs back to back: the second call
    # must not see anything the first left in the shared scratch array
    cases = [(512, 384, 160, 1), (1024, 256, 96, 2)]
    for K, N, M, seed in cases:
        g, w = _layer(exq, K, N, seed)
        x16 = synth.activations(M, K, seed=seed)
        x = torch.from_numpy(x16).cuda()
        ref = _with_workspace(exq, torch, w, x)
        got = _without(exq, torch, w, x)
        torch.cuda.synchronize()
        assert exq.exq_get_last_device_error() == 0
        ref64 = ref.float().cpu().numpy().astype(np.float64)
        got64 = got.float().cpu().numpy().astype(np.float64)
        check_matmul(got64, ref64, f"noalloc vs workspace K={K} N={N} M={M}")
        check_matmul(got64, O.matmul(x16, oracle_W_gptq(g)), f"noalloc vs oracle K={K} N={N} M={M}")


def test_noalloc_rejects_oversized_scratch(env):
    exq, torch = env
    _, w = _layer(exq, 512, 256, 3)
    M = exq.NOALLOC_SCRATCH_BYTES // (512 * 2) + 1        # M * K * 2 just above the limit
    x = torch.zeros(M, 512, dtype=torch.float16, device="cuda")
    y = torch.zeros(M, 256, dtype=torch.float16, device="cuda")
    with pytest.raises(exq.ExqError) as ei:
        exq.exq_gemm_noalloc(w, x, y)
    assert ei.value.status == exq.EXQ_ERR_UNSUPPORTED


def test_noalloc_without_permutation(env):
    exq, torch = env
    # an EXL2 layer stored in input-feature order needs no scratch; two calls
    # in a row, each against the workspace path and the oracle
    for K, N, M, seed in ((512, 256, 200, 4), (1024, 384, 64, 5)):
        e = exl2_case(K, N, bpw=4.0, permute=False, seed=seed)
        qw, off = exq.exq_pack_exl2(e.q, e.bits)
        w = exq.exl2_weight(qw, off, e.s, None, K, N)
        x16 = synth.activations(M, K, seed=seed)
        x = torch.from_numpy(x16).cuda()
        ref = _with_workspace(exq, torch, w, x)
        got = _without(exq, torch, w, x)
        torch.cuda.synchronize()
        assert exq.exq_get_last_device_error() == 0
        got64 = got.float().cpu().numpy().astype(np.float64)
        check_matmul(got64, ref.float().cpu().numpy().astype(np.float64), f"noalloc no-perm vs workspace K={K}")
        check_matmul(got64, O.matmul(x16, oracle_W_exl2(e)), f"noalloc no-perm vs oracle K={K}")


def test_noalloc_at_the_scratch_limit(env):
    exq, torch = env
    # M * K * 2 equal to the scratch size is accepted
    K, N = 512, 256
    M = exq.NOALLOC_SCRATCH_BYTES // (K * 2)
    g, w = _layer(exq, K, N, 6)
    x16 = synth.activations(M, K, seed=6)
    x = torch.from_numpy(x16).cuda()
    ref = _with_workspace(exq, torch, w, x)
    got = _without(exq, torch, w, x)
    torch.cuda.synchronize()
    assert exq.exq_get_last_device_error() == 0
    got64 = got.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isfinite(got64), np.ones_like(got64, dtype=bool))
    check_matmul(got64, ref.float().cpu().numpy().astype(np.float64), "noalloc at the limit vs workspace")
    rows = np.random.default_rng(6).choice(M, 64, replace=False)
    check_matmul(got64[rows], O.matmul(x16[rows], oracle_W_gptq(g)), "noalloc at the limit vs oracle (rows)")


def test_noalloc_allocates_nothing(env):
    exq, torch = env
    g, w = _layer(exq, 512, 384, 7)
    x = torch.from_numpy(synth.activations(128, 512, seed=7)).cuda()
    y = torch.empty(128, 384, dtype=torch.float16, device="cuda")
    exq.exq_gemm_noalloc(w, x, y)  # warmed up: module loaded, scratch address known
    torch.cuda.synchronize()
    before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
    for _ in range(3):
        exq.exq_gemm_noalloc(w, x, y)
    torch.cuda.synchronize()
    after = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
    assert exq.exq_get_last_device_error() == 0
    assert before == after, (before, after)
