"""CPU-side checks of the C ABI: the library loads without a GPU, exports
every symbol include/exq.h declares, its host packers match the oracle's
packers bit for bit, and host-side argument checks reject bad input before
anything reaches CUDA."""
from __future__ import annotations

import ctypes
import re
from pathlib import Path

import numpy as np
import pytest

import oracle as O
import synth

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def exq():
    import __graft_entry__
    __graft_entry__.build()
    import quantized_weight_exq_gb300 as m
    return m


def test_library_exports_every_declared_symbol(exq):
    header = "\n".join(p.read_text() for p in sorted((ROOT / "include").glob("*.h")))
    header = re.sub(r"/\*.*?\*/", "", header, flags=re.S)
    declared = set(re.findall(r"\b(exq_[a-z0-9_]+)\s*\(", header))
    assert declared == set(exq.EXPORTED), declared ^ set(exq.EXPORTED)
    lib = ctypes.CDLL(exq.library_path())
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings(exq):
    for s in range(5):
        assert exq.status_string(s) and "unknown" not in exq.status_string(s)
    assert "unknown" in exq.status_string(99)


@pytest.mark.parametrize("act_order,gs", [(False, 128), (True, 128), (True, 32), (False, 64)])
def test_pack_gptq_matches_oracle(exq, act_order, gs):
    g = synth.gptq_layer(512, 72, gs, act_order=act_order, seed=gs)
    qw, qz, perm = exq.exq_pack_gptq(g.q, g.z, g.g_idx, gs)
    oqw, oqz, _, operm = O.pack_gptq(g.q, g.z, g.s, g.g_idx, gs)
    assert np.array_equal(perm, operm)
    assert np.array_equal(qw, oqw)
    assert np.array_equal(qz, oqz)


def test_exl2_seg_word_off_matches_oracle(exq):
    bits = np.array([8, 2, 3, 6, 5, 4, 4, 2, 8], dtype=np.uint8)
    off = exq.exq_exl2_seg_word_off(bits)
    assert np.array_equal(off, O.exl2_seg_word_off(bits))
    assert off[0] == 0 and off[-1] == bits.sum()
    with pytest.raises(exq.ExqError):
        exq.exq_exl2_seg_word_off(np.array([4, 7], dtype=np.uint8))


def test_pack_exl2_matches_oracle(exq):
    for seed, bits in ((1, None), (2, np.array([8, 2, 3, 6, 5, 4] * 3))):
        e = synth.exl2_layer(32 * 18, 40, bpw=4.0, bits=bits, seed=seed)
        qw, off = exq.exq_pack_exl2(e.q, e.bits)
        oqw, ooff, _, _ = O.pack_exl2(e.q, e.bits, e.s, e.perm)
        assert np.array_equal(off, ooff)
        assert np.array_equal(qw, oqw)
        assert exq.exq_exl2_word_rows(e.bits) == int(e.bits.astype(int).sum())


def test_packers_reject_bad_input(exq):
    q = np.zeros((64, 8), np.uint8)
    z = np.zeros((2, 8), np.uint8)
    with pytest.raises(exq.ExqError):
        exq.exq_pack_gptq(np.full((64, 8), 16, np.uint8), z, None, 32)   # code > 15
    with pytest.raises(exq.ExqError):
        exq.exq_pack_gptq(q, z, np.array([0] * 33 + [1] * 31, np.int32), 32)  # unequal groups
    with pytest.raises(exq.ExqError):
        exq.exq_pack_gptq(q[:, :6], z[:, :6], None, 32)  # N % 8
    with pytest.raises(exq.ExqError):
        exq.exq_pack_exl2(np.full((64, 8), 4, np.uint8), np.array([2, 2], np.uint8))  # code too wide
    with pytest.raises(exq.ExqError):
        exq.exq_pack_exl2(q, np.array([2, 7], np.uint8))  # width outside the set
    assert exq.exq_exl2_word_rows(np.array([2, 7], np.uint8)) == -1


def _desc(exq, **kw):
    base = dict(format=exq.EXQ_FMT_GPTQ4, K=256, N=64, group_size=128, n_groups=2, n_word_rows=32,
                qweight=0x10000, scales=0x20000, qzeros=0x30000, perm=None, seg_word_off=None,
                q_scale=None, q_scale_max=None)
    base.update(kw)
    return exq.exq_weight(*[base[f] for f, _ in exq.exq_weight._fields_])


def test_device_entry_points_validate_on_host(exq):
    from quantized_weight_exq_gb300 import exq as mod
    lib = mod._lib
    bad = [
        dict(N=60),                        # N % 8
        dict(K=250),                       # K % 32
        dict(group_size=48),               # group % 32
        dict(n_groups=3),                  # inconsistent G
        dict(qweight=0x10004),             # misaligned
        dict(qzeros=None),                 # GPTQ without zeros
        dict(format=7),                    # unknown format
        dict(format=2, group_size=32, n_groups=8, n_word_rows=32, qzeros=None, seg_word_off=None),
        dict(format=2, group_size=32, n_groups=8, n_word_rows=100, qzeros=None, seg_word_off=0x40000),
    ]
    for kw in bad:
        d = _desc(exq, **kw)
        assert lib.exq_gemv(ctypes.byref(d), 0x50000, 1, 0x60000, None, 0, None) == exq.EXQ_ERR_INVALID_ARG, kw
        assert lib.exq_dequant(ctypes.byref(d), 0x60000, None) == exq.EXQ_ERR_INVALID_ARG, kw
        assert lib.exq_gemm(ctypes.byref(d), 0x50000, 1, 0x60000, None, 0, None) == exq.EXQ_ERR_INVALID_ARG, kw
    d = _desc(exq)
    assert lib.exq_gemv(ctypes.byref(d), 0x50000, 17, 0x60000, None, 0, None) == exq.EXQ_ERR_UNSUPPORTED
    assert lib.exq_gemv(ctypes.byref(d), 0x50000, 0, 0x60000, None, 0, None) == exq.EXQ_ERR_INVALID_ARG
    assert lib.exq_gemv(ctypes.byref(d), 0x50008, 1, 0x60000, None, 0, None) == exq.EXQ_ERR_INVALID_ARG
    assert lib.exq_gemv(None, 0x50000, 1, 0x60000, None, 0, None) == exq.EXQ_ERR_INVALID_ARG
    # the decode workspace size is 0 outside M = 1..16 and for a bad layer
    assert lib.exq_gemv_workspace_size(ctypes.byref(d), 17) == 0
    assert lib.exq_gemv_workspace_size(ctypes.byref(d), 0) == 0
    assert lib.exq_gemv_workspace_size(ctypes.byref(_desc(exq, N=60)), 1) == 0
    # act-order prefill needs a workspace for the gathered activations
    dp = _desc(exq, perm=0x70000)
    assert lib.exq_gemm_workspace_size(ctypes.byref(dp), 128) == 128 * 256 * 2
    assert lib.exq_gemm(ctypes.byref(dp), 0x50000, 128, 0x60000, None, 0, None) == exq.EXQ_ERR_INVALID_ARG


def test_gemv_multi_validates_on_host(exq):
    from quantized_weight_exq_gb300 import exq as mod
    lib = mod._lib

    def call(descs, M=1, ys=None, x=0x50000):
        arr = (exq.exq_weight * max(len(descs), 1))(*descs)
        ys = [0x60000 + 0x1000 * i for i in range(len(descs))] if ys is None else ys
        yp = (ctypes.c_void_p * max(len(ys), 1))(*ys)
        return lib.exq_gemv_multi(arr, len(descs), x, M, yp, None, 0, None)

    d = _desc(exq)
    assert call([]) == exq.EXQ_ERR_INVALID_ARG                                    # no layers
    assert call([d] * 5) == exq.EXQ_ERR_INVALID_ARG                               # more than EXQ_GEMV_MAX_LAYERS
    assert call([d, _desc(exq, K=512, n_groups=4, n_word_rows=64)]) == exq.EXQ_ERR_INVALID_ARG  # mixed K
    assert call([d, _desc(exq, group_size=64, n_groups=4)]) == exq.EXQ_ERR_INVALID_ARG          # mixed group size
    exl2 = _desc(exq, format=2, group_size=32, n_groups=8, n_word_rows=32, qzeros=None, seg_word_off=0x40000)
    assert call([d, exl2]) == exq.EXQ_ERR_INVALID_ARG                             # mixed formats
    assert call([d, _desc(exq, N=60)]) == exq.EXQ_ERR_INVALID_ARG                 # a bad layer
    assert call([d, d], ys=[0x60000, None]) == exq.EXQ_ERR_INVALID_ARG           # a missing output
    assert call([d, d], ys=[0x60000, 0x61008]) == exq.EXQ_ERR_INVALID_ARG        # a misaligned output
    assert call([d, d], x=0x50008) == exq.EXQ_ERR_INVALID_ARG
    assert call([d, d], M=0) == exq.EXQ_ERR_INVALID_ARG
    assert call([d, d], M=17) == exq.EXQ_ERR_UNSUPPORTED
    assert lib.exq_gemv_multi(None, 1, 0x50000, 1, None, None, 0, None) == exq.EXQ_ERR_INVALID_ARG
    arr = (exq.exq_weight * 2)(d, d)
    assert lib.exq_gemv_multi(arr, 2, 0x50000, 1, None, None, 0, None) == exq.EXQ_ERR_INVALID_ARG
    # the workspace size is 0 for an invalid group or M
    assert lib.exq_gemv_multi_workspace_size(arr, 5, 1) == 0
    assert lib.exq_gemv_multi_workspace_size(arr, 0, 1) == 0
    assert lib.exq_gemv_multi_workspace_size(arr, 2, 17) == 0
    mixed = (exq.exq_weight * 2)(d, exl2)
    assert lib.exq_gemv_multi_workspace_size(mixed, 2, 1) == 0


def test_pack_exl2_qscale_matches_oracle(exq):
    codes, _ = synth.exl2_qscale_draws(12, 40, seed=2)
    assert np.array_equal(exq.exq_pack_exl2_qscale(codes), O.pack_exl2_qscale(codes))
    with pytest.raises(exq.ExqError):
        exq.exq_pack_exl2_qscale(np.full((2, 8), 16, np.uint8))   # code > 15
    with pytest.raises(exq.ExqError):
        exq.exq_pack_exl2_qscale(np.zeros((2, 12), np.uint8))     # N % 8


def test_two_level_descriptor_rules(exq):
    from quantized_weight_exq_gb300 import exq as mod
    lib = mod._lib
    qs = dict(format=exq.EXQ_FMT_EXL2_QSCALE, group_size=32, n_groups=8, n_word_rows=32, qzeros=None,
              seg_word_off=0x40000, scales=None, q_scale=0x80000, q_scale_max=0x90000)
    bad = [
        dict(scales=0x20000),            # fp16 scales as well
        dict(q_scale=None),              # no codes
        dict(q_scale_max=None),          # no maxima
        dict(q_scale=0x80004),           # misaligned codes
        dict(q_scale_max=0x90002),       # misaligned maxima
        dict(seg_word_off=None),         # no segment table
    ]
    for kw in bad:
        d = _desc(exq, **{**qs, **kw})
        assert lib.exq_gemv(ctypes.byref(d), 0x50000, 1, 0x60000, None, 0, None) == exq.EXQ_ERR_INVALID_ARG, kw
        assert lib.exq_dequant(ctypes.byref(d), 0x60000, None) == exq.EXQ_ERR_INVALID_ARG, kw
        assert lib.exq_gemm(ctypes.byref(d), 0x50000, 1, 0x60000, None, 0, None) == exq.EXQ_ERR_INVALID_ARG, kw
    # codes or maxima on the other formats are rejected too
    for kw in (dict(q_scale=0x80000), dict(q_scale_max=0x90000)):
        d = _desc(exq, **kw)
        assert lib.exq_gemv(ctypes.byref(d), 0x50000, 1, 0x60000, None, 0, None) == exq.EXQ_ERR_INVALID_ARG, kw
    # a two-level layer and an fp16-scale EXL2 layer do not group
    e = _desc(exq, format=exq.EXQ_FMT_EXL2, group_size=32, n_groups=8, n_word_rows=32, qzeros=None,
              seg_word_off=0x40000)
    arr = (exq.exq_weight * 2)(_desc(exq, **qs), e)
    yp = (ctypes.c_void_p * 2)(0x60000, 0x61000)
    assert lib.exq_gemv_multi(arr, 2, 0x50000, 1, yp, None, 0, None) == exq.EXQ_ERR_INVALID_ARG


def test_kv_codec_validates_on_host(exq):
    from quantized_weight_exq_gb300 import exq as mod
    lib = mod._lib
    ok = dict(a=0x50000, G=4, D=128, bits=4, b=0x60000, c=0x70000)

    def q(**kw):
        d = {**ok, **kw}
        return lib.exq_kv_quantize(d["a"], d["G"], d["D"], d["bits"], d["b"], d["c"], None)

    def dq(**kw):
        d = {**ok, **kw}
        return lib.exq_kv_dequantize(d["a"], d["b"], d["G"], d["D"], d["bits"], d["c"], None)

    for f in (q, dq):
        assert f(D=96) == exq.EXQ_ERR_UNSUPPORTED
        assert f(D=512) == exq.EXQ_ERR_UNSUPPORTED
        assert f(bits=5) == exq.EXQ_ERR_UNSUPPORTED
        assert f(bits=2) == exq.EXQ_ERR_UNSUPPORTED
        assert f(G=-1) == exq.EXQ_ERR_INVALID_ARG
        assert f(a=None) == exq.EXQ_ERR_INVALID_ARG
        assert f(b=0x60008) == exq.EXQ_ERR_INVALID_ARG
        assert f(c=None) == exq.EXQ_ERR_INVALID_ARG
        assert f(G=0, a=None, b=None, c=None) == exq.EXQ_OK   # nothing to do, no launch


def test_solve_exl2_bits_matches_oracle(exq):
    err = np.array([[100, 50, 20, 10, 5, 1], [80, 70, 60, 50, 40, 30], [400, 100, 30, 10, 5, 2]], np.float64)
    for budget in (6, 8, 12, 13, 24):
        assert np.array_equal(exq.exq_solve_exl2_bits(err, budget), O.solve_exl2_bits(err, budget)), budget
    rng = np.random.default_rng(9)
    for S in (1, 7, 64, 300):
        # decreasing error curves with ties sprinkled in
        e = np.sort(rng.random((S, 6)) * rng.integers(1, 4, (S, 1)), axis=1)[:, ::-1].copy()
        e[::5] = e[0]
        for bpw in (2.0, 2.5, 3.3, 4.0, 5.1, 8.0):
            budget = int(round(bpw * S))
            assert np.array_equal(exq.exq_solve_exl2_bits(e, budget), O.solve_exl2_bits(e, budget)), (S, bpw)
    with pytest.raises(exq.ExqError):
        exq.exq_solve_exl2_bits(err, 5)


def test_convert_validates_on_host(exq):
    from quantized_weight_exq_gb300 import exq as mod
    lib = mod._lib
    assert lib.exq_measure_exl2_workspace_size(100, 64) == 0
    assert lib.exq_measure_exl2_workspace_size(64, 60) == 0
    ws = lib.exq_measure_exl2_workspace_size(64, 512)
    assert ws == 2 * 2 * 6 * 4                        # 2 segments x 2 column blocks x 6 widths, fp32
    assert lib.exq_measure_exl2(0x10000, None, 64, 512, 0x20000, 0x30000, ws - 4, None) == exq.EXQ_ERR_INVALID_ARG
    assert lib.exq_measure_exl2(0x10002, None, 64, 512, 0x20000, 0x30000, ws, None) == exq.EXQ_ERR_INVALID_ARG
    assert lib.exq_measure_exl2(0x10000, None, 60, 512, 0x20000, 0x30000, ws, None) == exq.EXQ_ERR_INVALID_ARG
    assert lib.exq_quantize_exl2(0x10000, None, 64, 512, None, 8, 0x20000, 0x30000, None) == exq.EXQ_ERR_INVALID_ARG
    assert lib.exq_quantize_exl2(0x10000, None, 64, 512, 0x40000, 3, 0x20000, 0x30000, None) == exq.EXQ_ERR_INVALID_ARG
    assert lib.exq_quantize_exl2(0x10000, 0x50004, 64, 512, 0x40000, 8, 0x20000, 0x30000, None) == exq.EXQ_ERR_INVALID_ARG
