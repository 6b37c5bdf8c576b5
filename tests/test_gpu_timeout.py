"""Failure detection on the GPU without a fault: the test hook of
include/exq_testing.h makes the producer of a GEMV / GEMM launch issue no
copies, so the consumers wait for data that never comes. Their waits are
bounded: they must give up, the call must end with EXQ_ERR_TIMEOUT in the
device error word, the context must stay usable, and the next normal call
(on a re-zeroed workspace) must match the oracle again."""
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
    yield exq, torch
    exq.exq_testing_starve(0)


def test_gemv_wait_runs_out_then_recovers(env):
    exq, torch = env
    e = exl2_case(1024, 496, bpw=4.0, seed=21)
    qw, off = exq.exq_pack_exl2(e.q, e.bits)
    w = exq.exl2_weight(qw, off, e.s, e.perm, e.K, e.N)
    x16 = synth.activations(1, e.K, seed=21)
    x = torch.from_numpy(x16).cuda()
    y = torch.full((1, e.N), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.zeros(exq.exq_gemv_workspace_size(w, 1), dtype=torch.uint8, device="cuda")
    assert exq.exq_get_last_device_error() == exq.EXQ_OK
    exq.exq_testing_starve(64)   # 64 rounds of at most 20 us each
    try:
        exq.exq_gemv(w, x, y, workspace=ws)
        assert exq.exq_get_last_device_error() == exq.EXQ_ERR_TIMEOUT
    finally:
        exq.exq_testing_starve(0)
    ws.zero_()
    exq.exq_gemv(w, x, y, workspace=ws)
    torch.cuda.synchronize()
    assert exq.exq_get_last_device_error() == exq.EXQ_OK
    check_matmul(y.float().cpu().numpy().astype(np.float64), O.matmul(x16, oracle_W_exl2(e)), "gemv after timeout")


def test_gemm_wait_runs_out_then_recovers(env):
    exq, torch = env
    g = gptq_case(512, 256, 128, act_order=True, seed=22)
    qw, qz, perm = exq.exq_pack_gptq(g.q, g.z, g.g_idx, g.group_size)
    w = exq.gptq_weight(qw, qz, g.s, perm, g.K, g.N, g.group_size)
    x16 = synth.activations(200, g.K, seed=22)
    x = torch.from_numpy(x16).cuda()
    y = torch.full((200, g.N), float("nan"), dtype=torch.float16, device="cuda")
    nws = exq.exq_gemm_workspace_size(w, 200)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device="cuda")
    assert exq.exq_get_last_device_error() == exq.EXQ_OK
    exq.exq_testing_starve(20000)
    try:
        exq.exq_gemm(w, x, y, ws)
        assert exq.exq_get_last_device_error() == exq.EXQ_ERR_TIMEOUT
    finally:
        exq.exq_testing_starve(0)
    exq.exq_gemm(w, x, y, ws)
    torch.cuda.synchronize()
    assert exq.exq_get_last_device_error() == exq.EXQ_OK
    check_matmul(y.float().cpu().numpy().astype(np.float64), O.matmul(x16, oracle_W_gptq(g)), "gemm after timeout")
