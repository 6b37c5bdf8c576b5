"""GPU parity of exq_gemv_multi -- several layers that read the same x, one
launch -- against the CPU oracle, layer by layer, through the C ABI. Same
tolerance as exq_gemv: max(2e-2, 1 fp16 ulp) element-wise and rel-L2 <= 1e-3
per output row."""
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


def _x(torch, x16):
    return torch.from_numpy(np.ascontiguousarray(x16)).cuda()


def _gptq_dev(exq, g):
    qw, qz, perm = exq.exq_pack_gptq(g.q, g.z, g.g_idx, g.group_size)
    has_perm = not np.array_equal(perm, np.arange(g.K))
    return exq.gptq_weight(qw, qz, g.s, perm if has_perm else None, g.K, g.N, g.group_size)


def _exl2_dev(exq, e):
    qw, off = exq.exq_pack_exl2(e.q, e.bits)
    return exq.exl2_weight(qw, off, e.s, e.perm, e.K, e.N)


def _multi(exq, torch, ws, x16, workspace=None):
    M = x16.shape[0]
    ys = [torch.full((M, w.N), float("nan"), dtype=torch.float16, device="cuda") for w in ws]
    exq.exq_gemv_multi(ws, _x(torch, x16), ys, workspace=workspace)
    torch.cuda.synchronize()
    assert exq.exq_get_last_device_error() == 0
    return [y.float().cpu().numpy().astype(np.float64) for y in ys]


def _exl2_group(exq, K, Ns, permute, bpw=4.0, seed=0):
    allowed = (2, 3, 4) if bpw < 3 else synth.EXL2_BITS
    cases = [exl2_case(K, N, bpw=bpw, allowed=allowed, permute=p, seed=seed + 17 * i)
             for i, (N, p) in enumerate(zip(Ns, permute))]
    return [_exl2_dev(exq, e) for e in cases], [oracle_W_exl2(e) for e in cases]


def _gptq_group(exq, K, Ns, gs, act, seed=0):
    cases = [gptq_case(K, N, gs, act_order=a, seed=seed + 17 * i) for i, (N, a) in enumerate(zip(Ns, act))]
    return [_gptq_dev(exq, g) for g in cases], [oracle_W_gptq(g) for g in cases]


# ---------------------------------------------------------------- small groups, full comparison

EXL2_GROUPS = [  # K, Ns, permute per layer, bpw
    (1024, (256, 64, 64), (True, True, True), 4.0),            # q, k, v
    (2048, (200, 8, 264, 136), (True, False, True, False), 2.5),  # four layers, ragged tiles, mixed permutations
    (512, (1000, 1000), (False, False), 4.0),                   # gate, up without permutations: no gather
]
GPTQ_GROUPS = [  # K, Ns, group size, act-order per layer
    (1024, (200, 72, 72), 128, (True, True, False)),
    (2048, (264, 264), 64, (False, False)),
    (512, (8, 520), 32, (True, True)),
]


@pytest.mark.parametrize("M", [1, 5, 16])
@pytest.mark.parametrize("K,Ns,perm,bpw", EXL2_GROUPS)
def test_multi_exl2(env, M, K, Ns, perm, bpw):
    exq, torch = env
    ws, refs = _exl2_group(exq, K, Ns, perm, bpw, seed=K)
    x = synth.activations(M, K, seed=M + 5)
    for i, (y, W) in enumerate(zip(_multi(exq, torch, ws, x), refs)):
        check_matmul(y, O.matmul(x, W), f"exl2 group K={K} layer {i} M={M}")


@pytest.mark.parametrize("M", [1, 9, 16])
@pytest.mark.parametrize("K,Ns,gs,act", GPTQ_GROUPS)
def test_multi_gptq(env, M, K, Ns, gs, act):
    exq, torch = env
    ws, refs = _gptq_group(exq, K, Ns, gs, act, seed=K)
    x = synth.activations(M, K, seed=M + 6)
    for i, (y, W) in enumerate(zip(_multi(exq, torch, ws, x), refs)):
        check_matmul(y, O.matmul(x, W), f"gptq group K={K} layer {i} M={M}")


@pytest.mark.parametrize("ctas", [1, 3, 37, 1000])
def test_multi_any_split_over_ctas(env, ctas, monkeypatch):
    # the layers' units form one list shared evenly by however many CTAs
    # run, so shares cross layer boundaries; every split gives the oracle's
    # result and leaves the counters at zero
    exq, torch = env
    monkeypatch.setenv("EXQ_GEMV_CTAS", str(ctas))
    groups = [_exl2_group(exq, 1024, (200, 64, 520), (True, False, True), seed=ctas),
              _gptq_group(exq, 1024, (136, 264), 128, (True, False), seed=ctas)]
    for ws, refs in groups:
        for M in (1, 9):
            x = synth.activations(M, 1024, seed=M + ctas)
            work = torch.zeros(exq.exq_gemv_multi_workspace_size(ws, M), dtype=torch.uint8, device="cuda")
            for i, (y, W) in enumerate(zip(_multi(exq, torch, ws, x, workspace=work), refs)):
                check_matmul(y, O.matmul(x, W), f"ctas={ctas} layer {i} M={M}")
            assert int(work[:65536].view(torch.int32).abs().sum()) == 0


def test_multi_of_one_is_gemv(env):
    # a group of one layer is exq_gemv itself: same plan, same bits
    exq, torch = env
    for w in (_exl2_dev(exq, exl2_case(2048, 264, seed=2)), _gptq_dev(exq, gptq_case(2048, 264, 64, True, seed=2))):
        for M in (1, 12):
            x = _x(torch, synth.activations(M, 2048, seed=M))
            y1 = torch.empty(M, w.N, dtype=torch.float16, device="cuda")
            exq.exq_gemv(w, x, y1)
            (y2,) = exq.exq_gemv_multi([w], x, [torch.empty_like(y1)])
            torch.cuda.synchronize()
            assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_multi_deterministic_and_shared_workspace(env):
    # grouped and single calls alternate on one stream with one workspace
    exq, torch = env
    ws, refs = _exl2_group(exq, 4096, (512, 128, 128), (True, True, True), seed=3)
    g = gptq_case(4096, 256, 128, act_order=True, seed=4)
    wg = _gptq_dev(exq, g)
    need = max(exq.exq_gemv_multi_workspace_size(ws, 4), exq.exq_gemv_workspace_size(wg, 4))
    work = torch.zeros(need, dtype=torch.uint8, device="cuda")
    x16 = synth.activations(4, 4096, seed=3)
    x = _x(torch, x16)
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(10):
            ys = [torch.empty(4, w.N, dtype=torch.float16, device="cuda") for w in ws]
            exq.exq_gemv_multi(ws, x, ys, workspace=work)
            yg = torch.empty(4, 256, dtype=torch.float16, device="cuda")
            exq.exq_gemv(wg, x, yg, workspace=work)
            outs.append((ys, yg))
    s.synchronize()
    assert exq.exq_get_last_device_error() == 0
    for ys, yg in outs[1:]:
        for a, b in zip(ys + [yg], outs[0][0] + [outs[0][1]]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for y, W in zip(outs[0][0], refs):
        check_matmul(y.float().cpu().numpy().astype(np.float64), O.matmul(x16, W), "shared ws")
    check_matmul(outs[0][1].float().cpu().numpy().astype(np.float64), O.matmul(x16, oracle_W_gptq(g)), "shared ws gptq")
    assert int(work[:65536].view(torch.int32).abs().sum()) == 0


def test_multi_rejects_mixed_groups(env):
    exq, torch = env
    a = _exl2_dev(exq, exl2_case(1024, 64, seed=1))
    b = _exl2_dev(exq, exl2_case(2048, 64, seed=1))
    c = _gptq_dev(exq, gptq_case(1024, 64, 128, seed=1))
    x = _x(torch, synth.activations(1, 1024))
    y = [torch.empty(1, 64, dtype=torch.float16, device="cuda") for _ in range(5)]
    for ws in ([a, b], [a, c], [a] * 5, []):
        with pytest.raises(exq.ExqError) as ei:
            exq.exq_gemv_multi(ws, x, y[:len(ws)])
        assert ei.value.status == exq.EXQ_ERR_INVALID_ARG


# ---------------------------------------------------------------- full-size groups, sampled columns

def _stream_layer(exq, K, N, lin, wid):
    # one linear of the 70B EXL2 4.0 decode stream (uniform packed words)
    S = K // 32
    bits = synth.solve_bit_mix(S, 4.0, synth.EXL2_BITS, synth.rng_for(0, wid, lin, 4))
    off = O.exl2_seg_word_off(bits)
    qw = synth.uniform_words(int(off[-1]) * N, seed=lin, workload=wid).reshape(-1, N)
    s = synth.fp16_uniform(synth.rng_for(0, wid, lin, 2), 0.002, 0.03, (S, N))
    perm = synth.rng_for(0, wid, lin, 5).permutation(K).astype(np.int32)
    cols = np.unique(np.concatenate([np.random.default_rng(N + lin).choice(N, 96, replace=False), [0, N - 1]]))
    W_ref = O.dequant_exl2(qw, off, bits, s.view(np.uint16), perm, cols=cols)
    return exq.exl2_weight(qw, off, s, perm, K, N), cols, W_ref


@pytest.mark.parametrize("names", [("q", "k", "v"), ("gate", "up")])
def test_decode_stream_70b_groups_sampled(env, names):
    exq, torch = env
    wid = synth.WORKLOAD_IDS["decode_stream_70b"]
    lin_ids = [list(synth.LLAMA2_70B_SHAPES).index(n) for n in names]
    K = synth.LLAMA2_70B_SHAPES[names[0]][0]
    layers = [_stream_layer(exq, K, synth.LLAMA2_70B_SHAPES[n][1], lin, wid) for n, lin in zip(names, lin_ids)]
    x = synth.activations(1, K, seed=8, workload=wid)
    ys = _multi(exq, torch, [w for w, _, _ in layers], x)
    for n, y, (_, cols, W_ref) in zip(names, ys, layers):
        check_matmul(y[:, cols], O.matmul(x, W_ref), f"70b group {names} layer {n}")


@pytest.mark.parametrize("M", [1, 8])
def test_gemv_multi_four_long_layers(env, M):
    exq, torch = env
    # four EXL2 layers with K = 28672 (the down projection's K): at M = 8 their
    # segment tables and a two-slot ring no longer fit half an SM, so the
    # one-set kernel runs one CTA per SM with a five-slot ring; at M = 1 two
    # CTAs share an SM. Both against the oracle.
    K = 28672
    ws, Ws = _exl2_group(exq, K, (128, 248, 64, 200), (True, True, False, True), seed=90 + M)
    x = synth.activations(M, K, seed=M + 90)
    ys = _multi(exq, torch, ws, x)
    for i, (y, W) in enumerate(zip(ys, Ws)):
        check_matmul(y, O.matmul(x, W), f"four long layers, layer {i}, M={M}")
