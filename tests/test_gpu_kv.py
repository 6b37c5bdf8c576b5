"""GPU parity of the quantized KV cache codec (Q4 / Q6 / Q8) against the CPU
oracle, through the C ABI: codes, scales and read-back values bit-exact."""
from __future__ import annotations

import numpy as np
import pytest

import oracle as O
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_exq_gb300 as exq
    torch.cuda.set_device(0)
    return exq, torch


def _groups(G, D, seed):
    """Seeded KV-like groups: N(0, 1) values times a per-group magnitude over
    2^-16 .. 2^6, plus special groups (zeros, -0, a zero scale, subnormal
    scales, the largest finite value, exact quotient ties)."""
    rng = synth.rng_for(seed, synth.WORKLOAD_IDS["test"], D, 0)
    x = (rng.standard_normal((G, D)) * np.exp2(rng.integers(-16, 7, (G, 1)))).astype(np.float16)
    x[0] = 0
    x[1] = np.float16(-0.0)
    x[2] = np.float16(2.0 ** -24)
    x[3, 7] = np.float16(65504.0)
    x[4] = (rng.standard_normal(D) * 2.0 ** -17).astype(np.float16)
    x[5] = 0
    x[5, :4] = np.array([1.0, 585 * 2.0 ** -13, -585 * 2.0 ** -13, 1755 * 2.0 ** -13], np.float16)
    return x


def _bits16(t):
    return t.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("bits", [4, 6, 8])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_kv_codec_bit_exact(env, D, bits):
    exq, torch = env
    x = _groups(1000 + D, D, seed=bits)
    xd = torch.from_numpy(x).cuda()
    codes, scales = exq.exq_kv_quantize(xd, bits)
    u_ref, s_ref = O.kv_quantize(x, bits)
    w_ref = O.kv_pack(u_ref, bits)
    torch.cuda.synchronize()
    assert np.array_equal(_bits16(scales), s_ref)
    assert np.array_equal(codes.cpu().numpy().view(np.uint32), w_ref)
    out = exq.exq_kv_dequantize(codes, scales, D, bits)
    torch.cuda.synchronize()
    assert np.array_equal(_bits16(out), O.kv_dequantize(w_ref, s_ref, bits, D))


def _tie_groups(G, D, bits, seed):
    """Groups whose quotients x / s are half-integers or one fp16 step away
    from one: the scale s0 = (1 + j/4) 2^e has three significant bits, the
    maximum qmax s0 is one of the values (so s = s0 exactly), and every other
    value is (k + 1/2) s0 for k in [-qmax, qmax - 1], exact in fp16, or its
    fp16 neighbour above or below. Every such value sits in the window where
    the write path takes the exact division, or just outside it."""
    rng = np.random.default_rng(seed)
    qmax = (1 << (bits - 1)) - 1
    s0 = (1 + rng.integers(0, 4, G) / 4) * np.exp2(rng.integers(-10, 3, G).astype(np.float64))
    k = rng.integers(-qmax, qmax, (G, D))
    x = ((k + 0.5) * s0[:, None]).astype(np.float16)
    assert np.array_equal(x.astype(np.float64), (k + 0.5) * s0[:, None])  # the ties are exact
    step = rng.integers(-1, 2, (G, D))                                       # -1, 0 or +1 fp16 step
    bits16 = x.view(np.uint16).astype(np.int64)
    sign = np.where(x < 0, -1, 1)
    x = (bits16 + step * sign).astype(np.uint16).view(np.float16)
    x[np.arange(G), rng.integers(0, D, G)] = (qmax * s0).astype(np.float16)
    assert np.array_equal(np.abs(x.astype(np.float64)).max(axis=1), qmax * s0)
    return x


@pytest.mark.parametrize("bits", [4, 6, 8])
def test_kv_quotient_ties_and_neighbours(env, bits):
    # the write path rounds x / s from a multiply by an approximate 1 / s and
    # takes the exact division only near half-integers; here nearly every
    # value is an exact tie (to even) or one fp16 step from one
    exq, torch = env
    x = _tie_groups(4096, 128, bits, seed=bits)
    codes, scales = exq.exq_kv_quantize(torch.from_numpy(x).cuda(), bits)
    u_ref, s_ref = O.kv_quantize(x, bits)
    torch.cuda.synchronize()
    assert np.array_equal(_bits16(scales), s_ref)
    assert np.array_equal(codes.cpu().numpy().view(np.uint32), O.kv_pack(u_ref, bits))


def test_kv_dequantize_of_oracle_codes(env):
    # the read path alone, on codes and scales written by the oracle
    exq, torch = env
    rng = np.random.default_rng(6)
    for bits in (4, 6, 8):
        u = rng.integers(0, 1 << bits, size=(333, 128)).astype(np.uint8)
        s = (rng.random(333) * 0.1).astype(np.float16).view(np.uint16)
        w = O.kv_pack(u, bits)
        out = exq.exq_kv_dequantize(torch.from_numpy(w.view(np.int32)).cuda(),
                                    torch.from_numpy(s.view(np.float16)).cuda(), 128, bits)
        torch.cuda.synchronize()
        assert np.array_equal(_bits16(out), O.kv_dequantize(w, s, bits, 128))


def test_kv_codec_empty_and_deterministic(env):
    exq, torch = env
    x = torch.empty(0, 128, dtype=torch.float16, device="cuda")
    codes, scales = exq.exq_kv_quantize(x, 4)
    assert codes.numel() == 0 and scales.numel() == 0
    xd = torch.from_numpy(_groups(64, 128, seed=1)).cuda()
    a = exq.exq_kv_quantize(xd, 6)
    b = exq.exq_kv_quantize(xd, 6)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))


def test_kv_cache_70b_slice_sampled(env):
    # one layer's K and V of the Llama-2-70B cache at 32K context (8 KV heads,
    # D = 128: 524,288 groups), quantised and read back at each width;
    # sampled groups against the oracle
    exq, torch = env
    G, D = 2 * 32768 * 8, 128
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7)
    xd = (torch.randn(G, D, device="cuda", generator=gen) *
          torch.exp2(torch.randint(-6, 3, (G, 1), device="cuda", generator=gen).float())).half()
    idx = np.unique(np.concatenate([np.random.default_rng(3).choice(G, 1500, replace=False), [0, G - 1]]))
    x_s = xd[torch.from_numpy(idx).cuda()].cpu().numpy()
    for bits in (4, 6, 8):
        codes, scales = exq.exq_kv_quantize(xd, bits)
        out = exq.exq_kv_dequantize(codes, scales, D, bits)
        torch.cuda.synchronize()
        u_ref, s_ref = O.kv_quantize(x_s, bits)
        w_ref = O.kv_pack(u_ref, bits)
        ii = torch.from_numpy(idx).cuda()
        assert np.array_equal(_bits16(scales[ii]), s_ref), bits
        assert np.array_equal(codes[ii].cpu().numpy().view(np.uint32), w_ref), bits
        assert np.array_equal(_bits16(out[ii]), O.kv_dequantize(w_ref, s_ref, bits, D)), bits
