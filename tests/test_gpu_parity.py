"""GPU parity of exq_dequant and exq_gemv against the CPU oracle, through the
C ABI. Dequant must be bit-exact; matmul within max(2e-2, 1 fp16 ulp)
element-wise and rel-L2 <= 1e-3 per output row."""
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


def _dequant(exq, torch, w):
    W = torch.full((w.K, w.N), float("nan"), dtype=torch.float16, device="cuda")
    exq.exq_dequant(w, W)
    torch.cuda.synchronize()
    return W.cpu().numpy().view(np.uint16)


def _gemv(exq, torch, w, x16, poison=True):
    M = x16.shape[0]
    y = torch.full((M, w.N), float("nan"), dtype=torch.float16, device="cuda")
    exq.exq_gemv(w, _x(torch, x16), y)
    torch.cuda.synchronize()
    assert exq.exq_get_last_device_error() == 0
    return y.float().cpu().numpy().astype(np.float64)


# ---------------------------------------------------------------- small, full comparison

GPTQ_SMALL = [  # K, N, gs, act_order
    (1024, 200, 128, False), (1024, 200, 128, True), (512, 64, 32, True), (2048, 136, 64, True),
    (256, 8, 128, False),
]
EXL2_SMALL = [  # K, N, bits / bpw, perm
    (1024, 200, 4.0, True), (32 * 6, 72, np.array([2, 3, 4, 5, 6, 8]), True),
    (32 * 12, 64, np.array([8, 8, 6, 6, 5, 5, 3, 3, 2, 2, 4, 4]), False), (2048, 264, 2.5, True),
]


@pytest.mark.parametrize("K,N,gs,act", GPTQ_SMALL)
def test_dequant_gptq_bit_exact(env, K, N, gs, act):
    exq, torch = env
    g = gptq_case(K, N, gs, act_order=act, seed=K + N)
    W = _dequant(exq, torch, _gptq_dev(exq, g))
    assert np.array_equal(W, oracle_W_gptq(g))


@pytest.mark.parametrize("K,N,bits,perm", EXL2_SMALL)
def test_dequant_exl2_bit_exact(env, K, N, bits, perm):
    exq, torch = env
    kw = dict(bits=bits) if isinstance(bits, np.ndarray) else dict(bpw=bits, allowed=(2, 3, 4) if bits < 3 else synth.EXL2_BITS)
    e = exl2_case(K, N, permute=perm, seed=K + N, **kw)
    W = _dequant(exq, torch, _exl2_dev(exq, e))
    assert np.array_equal(W, oracle_W_exl2(e))


def test_dequant_special_scales(env):
    # subnormal-producing, overflowing and negative scales, zero scales
    exq, torch = env
    K, N = 256, 64
    g = gptq_case(K, N, 128, seed=5)
    s = g.s.copy()
    s[0, :16] = np.float16(2.0 ** -20)
    s[0, 16:32] = np.float16(-5000.0)
    s[1, :16] = np.float16(-0.0)
    s[1, 16:32] = np.float16(-(2.0 ** -24))
    g.s = s
    W = _dequant(exq, torch, _gptq_dev(exq, g))
    assert np.array_equal(W, oracle_W_gptq(g))


@pytest.mark.parametrize("M", [1, 2, 5, 8, 9, 16])
@pytest.mark.parametrize("K,N,gs,act", GPTQ_SMALL[:4])
def test_gemv_gptq_small(env, M, K, N, gs, act):
    exq, torch = env
    g = gptq_case(K, N, gs, act_order=act, seed=K + N)
    x = synth.activations(M, K, seed=M)
    y = _gemv(exq, torch, _gptq_dev(exq, g), x)
    check_matmul(y, O.matmul(x, oracle_W_gptq(g)), f"gptq K={K} N={N} M={M}")


@pytest.mark.parametrize("M", [1, 3, 8, 16])
@pytest.mark.parametrize("K,N,bits,perm", EXL2_SMALL)
def test_gemv_exl2_small(env, M, K, N, bits, perm):
    exq, torch = env
    kw = dict(bits=bits) if isinstance(bits, np.ndarray) else dict(bpw=bits, allowed=(2, 3, 4) if bits < 3 else synth.EXL2_BITS)
    e = exl2_case(K, N, permute=perm, seed=K + N, **kw)
    x = synth.activations(M, K, seed=M + 100)
    y = _gemv(exq, torch, _exl2_dev(exq, e), x)
    check_matmul(y, O.matmul(x, oracle_W_exl2(e)), f"exl2 K={K} N={N} M={M}")


@pytest.mark.parametrize("rows", [32, 40])
@pytest.mark.parametrize("K,N,bits,perm", EXL2_SMALL + [(4096, 520, 3.0, True)])
def test_gemv_exl2_both_stage_heights(env, rows, K, N, bits, perm, monkeypatch):
    # EXL2 stages of 32 or 40 word rows: the one-set kernel (M <= 8) takes
    # 40 where two such slots fit half an SM, and the test hook keeps them at
    # 32; both on every SM and on 3 CTAs (several stages and pieces per CTA)
    exq, torch = env
    monkeypatch.setenv("EXQ_GEMV_ROWS", str(rows))
    kw = dict(bits=bits) if isinstance(bits, np.ndarray) else dict(bpw=bits, allowed=(2, 3, 4) if bits < 3 else synth.EXL2_BITS)
    e = exl2_case(K, N, permute=perm, seed=K + N + rows, **kw)
    w = _exl2_dev(exq, e)
    W_ref = oracle_W_exl2(e)
    for ctas in (None, 3):
        if ctas:
            monkeypatch.setenv("EXQ_GEMV_CTAS", str(ctas))
        for M in (1, 4):
            x = synth.activations(M, K, seed=M + rows)
            check_matmul(_gemv(exq, torch, w, x), O.matmul(x, W_ref), f"rows={rows} ctas={ctas} K={K} N={N} M={M}")


def test_gemv_one_hot_rows_exact(env):
    # x = e_k reproduces row k of the dequantized weight exactly (fp32 sum of
    # one product, rounded back to fp16)
    exq, torch = env
    for w_np, wdev in ((lambda g: (oracle_W_gptq(g), _gptq_dev(exq, g)))(gptq_case(1024, 136, 128, True, seed=9)),
                       (lambda e: (oracle_W_exl2(e), _exl2_dev(exq, e)))(exl2_case(1024, 136, seed=9))):
        ks = np.random.default_rng(1).choice(1024, 16, replace=False)
        x = np.zeros((16, 1024), np.float16)
        x[np.arange(16), ks] = 1.0
        y = _gemv(exq, torch, wdev, x)
        assert np.array_equal(y, O.float64_from_fp16_bits(w_np[ks]))


def test_gemv_deterministic_and_stream(env):
    exq, torch = env
    e = exl2_case(4096, 1024, seed=3)
    w = _exl2_dev(exq, e)
    x = _x(torch, synth.activations(4, 4096, seed=3))
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(20):
            y = torch.empty(4, 1024, dtype=torch.float16, device="cuda")
            exq.exq_gemv(w, x, y)
            outs.append(y)
    s.synchronize()
    for y in outs[1:]:
        assert torch.equal(y.view(torch.int16), outs[0].view(torch.int16))


def test_device_error_word_bad_segment(env):
    # a segment table whose widths are outside the set: the kernels skip those
    # segments (no access past the buffer) and report it on the host
    exq, torch = env
    e = exl2_case(256, 64, bits=np.array([4] * 8), permute=False, seed=4)
    qw, off = exq.exq_pack_exl2(e.q, e.bits)
    bad = off.copy()
    bad[1:] += 3                       # segment 0 -> width 7
    w = exq.exl2_weight(qw, bad, e.s, None, e.K, e.N)
    w.qweight = torch.zeros(int(bad[-1]), e.N, dtype=torch.int32, device="cuda")  # big enough
    w._desc = None
    y = torch.empty(1, e.N, dtype=torch.float16, device="cuda")
    exq.exq_gemv(w, _x(torch, synth.activations(1, 256)), y)
    assert exq.exq_get_last_device_error() == exq.EXQ_ERR_INVALID_ARG
    assert exq.exq_get_last_device_error() == 0  # read-and-clear


@pytest.mark.parametrize("ctas", [1, 2, 5, 37, 1000])
def test_gemv_any_split_over_ctas(env, ctas, monkeypatch):
    # the (tile, step) work is shared evenly by however many CTAs run; tiles
    # split between CTAs meet in the workspace. Every split gives the oracle's
    # result, and every call leaves the workspace counters at zero.
    exq, torch = env
    monkeypatch.setenv("EXQ_GEMV_CTAS", str(ctas))
    g = gptq_case(2048, 264, 64, act_order=True, seed=ctas)
    e = exl2_case(2048, 200, bpw=4.0, permute=True, seed=ctas)
    for w, W_ref in ((_gptq_dev(exq, g), oracle_W_gptq(g)), (_exl2_dev(exq, e), oracle_W_exl2(e))):
        for M in (1, 9):
            x = synth.activations(M, w.K, seed=M + ctas)
            ws = torch.zeros(exq.exq_gemv_workspace_size(w, M), dtype=torch.uint8, device="cuda")
            y = torch.full((M, w.N), float("nan"), dtype=torch.float16, device="cuda")
            exq.exq_gemv(w, _x(torch, x), y, workspace=ws)
            torch.cuda.synchronize()
            assert exq.exq_get_last_device_error() == 0
            assert int(ws[:65536].view(torch.int32).abs().sum()) == 0  # the counters are zero again
            check_matmul(y.float().cpu().numpy().astype(np.float64), O.matmul(x, W_ref), f"ctas={ctas} M={M}")


def test_gemv_workspace_contract(env):
    exq, torch = env
    e = exl2_case(1024, 128, seed=11)
    w = _exl2_dev(exq, e)
    need = exq.exq_gemv_workspace_size(w, 1)
    assert need > 0
    x = _x(torch, synth.activations(1, 1024, seed=1))
    y = torch.empty(1, 128, dtype=torch.float16, device="cuda")
    short = torch.zeros(need - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(exq.ExqError) as ei:
        exq.exq_gemv(w, x, y, workspace=short)
    assert ei.value.status == exq.EXQ_ERR_INVALID_ARG
    # one workspace, as large as the largest call needs, serves a run of
    # calls with different layers and M
    runs = [(K, N, M, exl2_case(K, N, seed=K + M)) for K, N, M in ((1024, 128, 1), (4096, 1024, 16), (2048, 264, 3))]
    devs = [_exl2_dev(exq, ee) for _, _, _, ee in runs]
    ws = torch.zeros(max(exq.exq_gemv_workspace_size(ww, M) for (_, _, M, _), ww in zip(runs, devs)),
                     dtype=torch.uint8, device="cuda")
    for (K, N, M, ee), ww in zip(runs, devs):
        xx = synth.activations(M, K, seed=M)
        yy = torch.empty(M, N, dtype=torch.float16, device="cuda")
        exq.exq_gemv(ww, _x(torch, xx), yy, workspace=ws)
        torch.cuda.synchronize()
        check_matmul(yy.float().cpu().numpy().astype(np.float64), O.matmul(xx, oracle_W_exl2(ee)), f"ws K={K} M={M}")
    assert int(ws[:65536].view(torch.int32).abs().sum()) == 0  # the counter region is zero again


# ---------------------------------------------------------------- full-size workloads

def _sample_cols(N, n=256, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.choice(N, n, replace=False), [0, N - 1]]))


def test_gptq_gemv_4096(env):
    # M=1, K=N=4096, group 128, no act-order: full comparison
    exq, torch = env
    g = gptq_case(4096, 4096, 128, act_order=False, seed=0, workload=synth.WORKLOAD_IDS["gptq_gemv_4096"])
    w = _gptq_dev(exq, g)
    x = synth.activations(1, 4096, seed=0, workload=synth.WORKLOAD_IDS["gptq_gemv_4096"])
    W_ref = oracle_W_gptq(g)
    assert np.array_equal(_dequant(exq, torch, w), W_ref)
    check_matmul(_gemv(exq, torch, w, x), O.matmul(x, W_ref), "gptq 4096")


@pytest.mark.parametrize("name", ["q", "gate", "down"])
def test_gptq_act_order_7b(env, name):
    exq, torch = env
    K, N = synth.LLAMA2_7B_SHAPES[name]
    wid = synth.WORKLOAD_IDS["gptq_act_order_7b"]
    g = gptq_case(K, N, 128, act_order=True, seed=0, workload=wid, layer=list(synth.LLAMA2_7B_SHAPES).index(name))
    w = _gptq_dev(exq, g)
    cols = _sample_cols(N, seed=K)
    W_ref = oracle_W_gptq(g, cols=cols)
    assert np.array_equal(_dequant(exq, torch, w)[:, cols], W_ref)
    for M in (1, 4, 16):
        x = synth.activations(M, K, seed=M, workload=wid)
        check_matmul(_gemv(exq, torch, w, x)[:, cols], O.matmul(x, W_ref), f"gptq7b {name} M={M}")


@pytest.mark.parametrize("name", ["k", "up", "down"])
def test_exl2_4p0_7b(env, name):
    exq, torch = env
    K, N = synth.LLAMA2_7B_SHAPES[name]
    wid = synth.WORKLOAD_IDS["exl2_4p0_7b"]
    e = exl2_case(K, N, bpw=4.0, seed=0, workload=wid, layer=list(synth.LLAMA2_7B_SHAPES).index(name))
    w = _exl2_dev(exq, e)
    cols = _sample_cols(N, seed=K + 1)
    W_ref = oracle_W_exl2(e, cols=cols)
    assert np.array_equal(_dequant(exq, torch, w)[:, cols], W_ref)
    for M in (1, 8):
        x = synth.activations(M, K, seed=M, workload=wid)
        check_matmul(_gemv(exq, torch, w, x)[:, cols], O.matmul(x, W_ref), f"exl2 7b {name} M={M}")


@pytest.mark.parametrize("name", ["k", "gate", "down"])
def test_decode_stream_70b_sampled(env, name):
    # the 70B EXL2 4.0 stream draws its packed words uniformly (a packed
    # segment column is a bijection of 32 uniform codes)
    exq, torch = env
    K, N = synth.LLAMA2_70B_SHAPES[name]
    wid = synth.WORKLOAD_IDS["decode_stream_70b"]
    S = K // 32
    bits = synth.solve_bit_mix(S, 4.0, synth.EXL2_BITS, synth.rng_for(0, wid, 0, 4))
    off = O.exl2_seg_word_off(bits)
    qw = synth.uniform_words(int(off[-1]) * N, seed=0, workload=wid).reshape(-1, N)
    s = synth.fp16_uniform(synth.rng_for(0, wid, 0, 2), 0.002, 0.03, (S, N))
    perm = synth.rng_for(0, wid, 0, 5).permutation(K).astype(np.int32)
    w = exq.exl2_weight(qw, off, s, perm, K, N)
    cols = _sample_cols(N, n=128, seed=N)
    W_ref = O.dequant_exl2(qw, off, bits, s.view(np.uint16), perm, cols=cols)
    assert np.array_equal(_dequant(exq, torch, w)[:, cols], W_ref)
    x = synth.activations(1, K, seed=7, workload=wid)
    check_matmul(_gemv(exq, torch, w, x)[:, cols], O.matmul(x, W_ref), f"70b {name}")


# ---------------------------------------------------------------- size limits and degenerate shapes

def test_gemv_single_segment(env):
    # K = 32: one segment, one stage, every CTA but one idle
    exq, torch = env
    for bits in (np.array([2]), np.array([3]), np.array([8])):
        e = exl2_case(32, 200, bits=bits, permute=True, seed=int(bits[0]))
        for M in (1, 16):
            x = synth.activations(M, 32, seed=M)
            check_matmul(_gemv(exq, torch, _exl2_dev(exq, e), x), O.matmul(x, oracle_W_exl2(e)), f"K=32 b={bits}")
    g = gptq_case(32, 64, 32, act_order=True, seed=2)
    x = synth.activations(3, 32, seed=3)
    check_matmul(_gemv(exq, torch, _gptq_dev(exq, g), x), O.matmul(x, oracle_W_gptq(g)), "gptq K=32")


def test_gemv_widest_layer(env):
    # the most columns one call takes: 2048 tiles of 248 (N = 507,904), K = 64;
    # sampled columns against the oracle, the last tile included
    exq, torch = env
    N = 2048 * 248
    e = exl2_case(64, N, bits=np.array([4, 6]), permute=False, seed=5)
    w = _exl2_dev(exq, e)
    x = synth.activations(1, 64, seed=5)
    cols = np.unique(np.concatenate([np.random.default_rng(5).choice(N, 300, replace=False), np.arange(N - 300, N)]))
    check_matmul(_gemv(exq, torch, w, x)[:, cols], O.matmul(x, oracle_W_exl2(e, cols=cols)), "N = 507904")
    # one more tile is past the counter region
    e2 = exl2_case(64, N + 8, bits=np.array([4, 4]), permute=False, seed=6)
    assert exq.exq_gemv_workspace_size(_exl2_dev(exq, e2), 1) == 0


def test_gemv_deepest_layer(env):
    # the longest K segment indices allow: 65535 segments (K = 2,097,120), N = 8
    exq, torch = env
    K = 65535 * 32
    g = gptq_case(K, 8, 32, act_order=False, seed=7)
    w = _gptq_dev(exq, g)
    x = synth.activations(1, K, seed=7)
    check_matmul(_gemv(exq, torch, w, x), O.matmul(x, oracle_W_gptq(g)), "K = 2097120")
    g2 = gptq_case(K + 32, 8, 32, act_order=False, seed=8)
    assert exq.exq_gemv_workspace_size(_gptq_dev(exq, g2), 1) == 0
