"""Python binding of libexq (ctypes): argument marshalling only.

Every function here forwards to the C ABI in ``include/exq.h`` with the same
name; all arithmetic runs in the library (host packers in C++, device ops in
CUDA kernels). torch is used only to hold device memory and to name the
current CUDA stream. If ``libexq.so`` has not been built, importing this
module raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field
from pathlib import Path
from typing import Optional

import numpy as np

_LIB_PATH = Path(__file__).resolve().parent / "libexq.so"

EXQ_OK = 0
EXQ_ERR_INVALID_ARG = 1
EXQ_ERR_UNSUPPORTED = 2
EXQ_ERR_CUDA = 3
EXQ_ERR_TIMEOUT = 4

EXQ_FMT_GPTQ4 = 1
EXQ_FMT_EXL2 = 2
EXQ_FMT_EXL2_QSCALE = 3

# every symbol include/exq.h declares
EXPORTED = (
    "exq_pack_gptq", "exq_pack_exl2", "exq_pack_exl2_qscale", "exq_exl2_word_rows", "exq_exl2_seg_word_off",
    "exq_dequant", "exq_gemv_workspace_size",
    "exq_gemv", "exq_gemv_multi_workspace_size", "exq_gemv_multi", "exq_gemm_workspace_size", "exq_gemm", "exq_gemm_multi_workspace_size", "exq_gemm_multi", "exq_gemm_noalloc", "exq_status_string",
    "exq_get_last_device_error", "exq_kv_quantize", "exq_kv_dequantize",
    "exq_quantize_exl2", "exq_measure_exl2_workspace_size", "exq_measure_exl2", "exq_solve_exl2_bits",
    "exq_testing_starve",
)

# most layers one exq_gemv_multi call takes (EXQ_GEMV_MAX_LAYERS)
GEMV_MAX_LAYERS = 4

# size of the static scratch array exq_gemm_noalloc uses (EXQ_NOALLOC_SCRATCH_BYTES)
NOALLOC_SCRATCH_BYTES = 16 << 20


class ExqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class exq_weight(ctypes.Structure):
    _fields_ = [
        ("format", ctypes.c_int32), ("K", ctypes.c_int32), ("N", ctypes.c_int32),
        ("group_size", ctypes.c_int32), ("n_groups", ctypes.c_int32), ("n_word_rows", ctypes.c_int32),
        ("qweight", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("qzeros", ctypes.c_void_p),
        ("perm", ctypes.c_void_p), ("seg_word_off", ctypes.c_void_p),
        ("q_scale", ctypes.c_void_p), ("q_scale_max", ctypes.c_void_p),
    ]


def _load():
    if not _LIB_PATH.exists():
        raise ImportError(f"{_LIB_PATH} is not built; run quantized_weight_exq_gb300/build.py "
                          "(or __graft_entry__.build())")
    lib = ctypes.CDLL(str(_LIB_PATH))
    P, i32, i64, sz, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
    W = ctypes.POINTER(exq_weight)
    sig = {
        "exq_pack_gptq": (st, [P, P, P, i32, i32, i32, P, P, P]),
        "exq_pack_exl2": (st, [P, P, i32, i32, P, P]),
        "exq_pack_exl2_qscale": (st, [P, i32, i32, P]),
        "exq_exl2_word_rows": (i64, [P, i32]),
        "exq_exl2_seg_word_off": (st, [P, i32, P]),
        "exq_dequant": (st, [W, P, P]),
        "exq_gemv_workspace_size": (sz, [W, i32]),
        "exq_gemv": (st, [W, P, i32, P, P, sz, P]),
        "exq_gemv_multi_workspace_size": (sz, [W, i32, i32]),
        "exq_gemv_multi": (st, [W, i32, P, i32, P, P, sz, P]),
        "exq_gemm_workspace_size": (sz, [W, i32]),
        "exq_gemm": (st, [W, P, i32, P, P, sz, P]),
        "exq_gemm_noalloc": (st, [W, P, i32, P, P]),
        "exq_gemm_multi_workspace_size": (sz, [W, i32, i32]),
        "exq_gemm_multi": (st, [W, i32, P, i32, P, P, sz, P]),
        "exq_kv_quantize": (st, [P, i64, i32, i32, P, P, P]),
        "exq_kv_dequantize": (st, [P, P, i64, i32, i32, P, P]),
        "exq_quantize_exl2": (st, [P, P, i32, i32, P, i32, P, P, P]),
        "exq_measure_exl2_workspace_size": (sz, [i32, i32]),
        "exq_measure_exl2": (st, [P, P, i32, i32, P, P, sz, P]),
        "exq_solve_exl2_bits": (st, [P, i32, i64, P]),
        "exq_status_string": (ctypes.c_char_p, [st]),
        "exq_get_last_device_error": (st, [P]),
        "exq_testing_starve": (None, [i32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def library_path() -> str:
    return str(_LIB_PATH)


def status_string(status: int) -> str:
    return _lib.exq_status_string(int(status)).decode()


exq_status_string = status_string


def _check(status: int, where: str):
    if status != EXQ_OK:
        raise ExqError(status, where)


def _np_ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------- host packers

def exq_pack_gptq(q: np.ndarray, z: np.ndarray, g_idx: Optional[np.ndarray], group_size: int):
    """-> (qweight uint32 [K/8, N], qzeros uint32 [G, N/8], perm int32 [K])."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    K, N = q.shape
    gi = None if g_idx is None else np.ascontiguousarray(g_idx, dtype=np.int32)
    qweight = np.empty((K // 8, N), dtype=np.uint32)
    qzeros = np.empty((max(K // max(group_size, 1), 1), N // 8), dtype=np.uint32)
    perm = np.empty(K, dtype=np.int32)
    _check(_lib.exq_pack_gptq(_np_ptr(q), _np_ptr(z), _np_ptr(gi), K, N, group_size,
                              _np_ptr(qweight), _np_ptr(qzeros), _np_ptr(perm)), "exq_pack_gptq")
    return qweight, qzeros, perm


def exq_exl2_word_rows(bits: np.ndarray) -> int:
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    return int(_lib.exq_exl2_word_rows(_np_ptr(bits), bits.size))


def exq_exl2_seg_word_off(bits: np.ndarray) -> np.ndarray:
    """Segment table uint32 [S + 1] (word-row prefix sums) of the widths [S]."""
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    off = np.empty(bits.size + 1, dtype=np.uint32)
    _check(_lib.exq_exl2_seg_word_off(_np_ptr(bits), bits.size, _np_ptr(off)), "exq_exl2_seg_word_off")
    return off


def exq_pack_exl2(q: np.ndarray, bits: np.ndarray):
    """-> (qweight uint32 [sum(bits), N], seg_word_off uint32 [S + 1])."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    bits = np.ascontiguousarray(bits, dtype=np.uint8)
    K, N = q.shape
    rows = exq_exl2_word_rows(bits)
    if rows < 0:
        raise ExqError(EXQ_ERR_INVALID_ARG, "exq_pack_exl2")
    qweight = np.empty((rows, N), dtype=np.uint32)
    off = np.empty(bits.size + 1, dtype=np.uint32)
    _check(_lib.exq_pack_exl2(_np_ptr(q), _np_ptr(bits), K, N, _np_ptr(qweight), _np_ptr(off)), "exq_pack_exl2")
    return qweight, off


def exq_pack_exl2_qscale(codes: np.ndarray) -> np.ndarray:
    """4-bit scale codes uint8 [S, N] -> q_scale uint32 [S, N/8]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    S, N = codes.shape
    out = np.empty((S, max(N // 8, 1)), dtype=np.uint32)
    _check(_lib.exq_pack_exl2_qscale(_np_ptr(codes), S, N, _np_ptr(out)), "exq_pack_exl2_qscale")
    return out


# ---------------------------------------------------------------- device layer

@dataclass
class Weight:
    """A packed layer resident on the GPU (torch tensors hold the memory)."""

    format: int
    K: int
    N: int
    group_size: int
    qweight: "object"                 # torch.int32 [rows, N] (uint32 bits)
    scales: "object"                  # torch.float16 [G or S, N]; None for EXL2 two-level
    qzeros: "object" = None           # torch.int32 [G, N/8] (GPTQ)
    perm: "object" = None             # torch.int32 [K]
    seg_word_off: "object" = None     # torch.int32 [S + 1] (EXL2)
    q_scale: "object" = None          # torch.int32 [S, N/8] 4-bit codes (EXL2 two-level)
    q_scale_max: "object" = None      # torch.float16 [N] (EXL2 two-level)
    _desc: exq_weight = field(default=None, repr=False)

    def desc(self) -> exq_weight:
        if self._desc is None:
            ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
            groups = self.scales.shape[0] if self.scales is not None else self.q_scale.shape[0]
            self._desc = exq_weight(
                self.format, self.K, self.N, self.group_size, groups, self.qweight.shape[0],
                ptr(self.qweight), ptr(self.scales), ptr(self.qzeros), ptr(self.perm), ptr(self.seg_word_off),
                ptr(self.q_scale), ptr(self.q_scale_max))
        return self._desc

    @property
    def packed_bytes(self) -> int:
        """qweight + scales (or scale codes and column maxima) + qzeros bytes:
        the weight stream of one matmul."""
        n = self.qweight.numel() * 4
        for t, size in ((self.scales, 2), (self.qzeros, 4), (self.q_scale, 4), (self.q_scale_max, 2)):
            if t is not None:
                n += t.numel() * size
        return n


def _dev(a, dtype, device):
    import torch
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        return a.to(device=device).contiguous()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    if a.dtype == np.uint16:
        a = a.view(np.float16)
    return torch.from_numpy(a).to(device=device, dtype=dtype).contiguous()


def gptq_weight(qweight, qzeros, scales, perm, K: int, N: int, group_size: int, device="cuda") -> Weight:
    import torch
    return Weight(EXQ_FMT_GPTQ4, K, N, group_size, _dev(qweight, torch.int32, device),
                  _dev(scales, torch.float16, device), _dev(qzeros, torch.int32, device),
                  _dev(perm, torch.int32, device), None)


def exl2_weight(qweight, seg_word_off, scales, perm, K: int, N: int, device="cuda") -> Weight:
    import torch
    return Weight(EXQ_FMT_EXL2, K, N, 32, _dev(qweight, torch.int32, device),
                  _dev(scales, torch.float16, device), None, _dev(perm, torch.int32, device),
                  _dev(seg_word_off, torch.int32, device))


def exl2_qscale_weight(qweight, seg_word_off, q_scale, q_scale_max, perm, K: int, N: int, device="cuda") -> Weight:
    """EXL2 layer with two-level scales: q_scale uint32 [S, N/8] packed codes
    (exq_pack_exl2_qscale), q_scale_max fp16 [N]."""
    import torch
    return Weight(EXQ_FMT_EXL2_QSCALE, K, N, 32, _dev(qweight, torch.int32, device), None, None,
                  _dev(perm, torch.int32, device), _dev(seg_word_off, torch.int32, device),
                  _dev(q_scale, torch.int32, device), _dev(q_scale_max, torch.float16, device))


def exq_dequant(w: Weight, W_out, stream=None):
    _check(_lib.exq_dequant(ctypes.byref(w.desc()), W_out.data_ptr(), _stream_ptr(stream)), "exq_dequant")
    return W_out


def exq_gemv_workspace_size(w: Weight, M: int) -> int:
    return int(_lib.exq_gemv_workspace_size(ctypes.byref(w.desc()), M))


_gemv_ws = {}  # device index -> zero-filled uint8 workspace shared by calls on one stream


def gemv_workspace(w: Weight, M: int):
    """A zero-filled exq_gemv workspace for the current device, kept and grown
    across calls. exq_gemv leaves it zeroed, so calls ordered on one stream can
    share it; calls that may overlap on the GPU need their own (torch.zeros of
    exq_gemv_workspace_size bytes)."""
    return _shared_workspace(exq_gemv_workspace_size(w, M))


def _shared_workspace(need: int):
    import torch
    dev = torch.cuda.current_device()
    buf = _gemv_ws.get(dev)
    if buf is None or buf.numel() < need:
        buf = torch.zeros(max(need, 1 << 20), dtype=torch.uint8, device=f"cuda:{dev}")
        _gemv_ws[dev] = buf
    return buf


def exq_gemv(w: Weight, x, y, workspace=None, stream=None):
    if workspace is None:
        workspace = gemv_workspace(w, x.shape[0])
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.exq_gemv(ctypes.byref(w.desc()), x.data_ptr(), x.shape[0], y.data_ptr(), workspace.data_ptr(),
                         ws_bytes, _stream_ptr(stream)), "exq_gemv")
    return y


def _desc_array(ws):
    return (exq_weight * len(ws))(*[w.desc() for w in ws])


def exq_gemv_multi_workspace_size(ws, M: int) -> int:
    return int(_lib.exq_gemv_multi_workspace_size(_desc_array(ws), len(ws), M))


def exq_gemv_multi(ws, x, ys, workspace=None, stream=None):
    """y_i = x . dequant(ws[i]) for the layers ws (one format, one K), in one
    launch. ``ys`` are the outputs, one per layer."""
    if len(ws) != len(ys):
        raise ExqError(EXQ_ERR_INVALID_ARG, "exq_gemv_multi")
    if workspace is None:
        workspace = _shared_workspace(exq_gemv_multi_workspace_size(ws, x.shape[0]))
    ws_bytes = workspace.numel() * workspace.element_size()
    yp = (ctypes.c_void_p * len(ys))(*[y.data_ptr() for y in ys])
    _check(_lib.exq_gemv_multi(_desc_array(ws), len(ws), x.data_ptr(), x.shape[0], yp, workspace.data_ptr(),
                               ws_bytes, _stream_ptr(stream)), "exq_gemv_multi")
    return ys


def exq_gemm_workspace_size(w: Weight, M: int) -> int:
    return int(_lib.exq_gemm_workspace_size(ctypes.byref(w.desc()), M))


def exq_gemm(w: Weight, x, y, workspace=None, stream=None):
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.exq_gemm(ctypes.byref(w.desc()), x.data_ptr(), x.shape[0], y.data_ptr(), ws_ptr, ws_bytes,
                         _stream_ptr(stream)), "exq_gemm")
    return y


def exq_gemm_multi_workspace_size(ws, M: int) -> int:
    return int(_lib.exq_gemm_multi_workspace_size(_desc_array(ws), len(ws), M))


def exq_gemm_multi(ws, x, ys, workspace=None, stream=None):
    """y_i = x . dequant(ws[i]) for the layers ws (one format, one K), in one
    prefill launch. ``ys`` are the outputs, one per layer."""
    import torch
    if len(ws) != len(ys):
        raise ExqError(EXQ_ERR_INVALID_ARG, "exq_gemm_multi")
    need = exq_gemm_multi_workspace_size(ws, x.shape[0])
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_ptr = None if workspace is None else workspace.data_ptr()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    yp = (ctypes.c_void_p * len(ys))(*[y.data_ptr() for y in ys])
    _check(_lib.exq_gemm_multi(_desc_array(ws), len(ws), x.data_ptr(), x.shape[0], yp, ws_ptr, ws_bytes,
                               _stream_ptr(stream)), "exq_gemm_multi")
    return ys


GEMM_MAX_LAYERS = 4


def exq_gemm_noalloc(w: Weight, x, y, stream=None):
    """exq_gemm for callers that cannot allocate: an act-order layer's
    gathered activations go to the library's static scratch array (see
    include/exq.h for the size limit, the first-call set-up and the rule that
    overlapping calls race on the shared array)."""
    _check(_lib.exq_gemm_noalloc(ctypes.byref(w.desc()), x.data_ptr(), x.shape[0], y.data_ptr(),
                                 _stream_ptr(stream)), "exq_gemm_noalloc")
    return y


def exq_kv_quantize(x, bits: int, codes=None, scales=None, stream=None):
    """Quantized KV cache write: x fp16 [..., D] (groups of D values) ->
    (codes int32 [groups, D * bits / 32] holding uint32 words, scales fp16 [groups])."""
    import torch
    D = x.shape[-1]
    G = x.numel() // D if D else 0
    if codes is None:
        codes = torch.empty(G, D * bits // 32, dtype=torch.int32, device=x.device)
    if scales is None:
        scales = torch.empty(G, dtype=torch.float16, device=x.device)
    _check(_lib.exq_kv_quantize(x.data_ptr(), G, D, bits, codes.data_ptr(), scales.data_ptr(), _stream_ptr(stream)),
           "exq_kv_quantize")
    return codes, scales


def exq_kv_dequantize(codes, scales, D: int, bits: int, out=None, stream=None):
    """Quantized KV cache read: fp16 [groups, D]."""
    import torch
    G = scales.numel()
    if out is None:
        out = torch.empty(G, D, dtype=torch.float16, device=scales.device)
    _check(_lib.exq_kv_dequantize(codes.data_ptr(), scales.data_ptr(), G, D, bits, out.data_ptr(),
                                  _stream_ptr(stream)), "exq_kv_dequantize")
    return out


def exq_solve_exl2_bits(err: np.ndarray, budget: int) -> np.ndarray:
    """Host: widths uint8 [S] for an error table float64 [S, 6] and a budget of
    code bits per column."""
    err = np.ascontiguousarray(err, dtype=np.float64)
    S = err.shape[0]
    out = np.empty(S, dtype=np.uint8)
    _check(_lib.exq_solve_exl2_bits(_np_ptr(err), S, int(budget), _np_ptr(out)), "exq_solve_exl2_bits")
    return out


def exq_measure_exl2(W, perm=None, stream=None):
    """RTN error table fp32 [K/32, 6] of an fp16 weight [K, N] (device)."""
    import torch
    K, N = W.shape
    err = torch.empty(K // 32, 6, dtype=torch.float32, device=W.device)
    nws = int(_lib.exq_measure_exl2_workspace_size(K, N))
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=W.device)
    _check(_lib.exq_measure_exl2(W.data_ptr(), None if perm is None else perm.data_ptr(), K, N, err.data_ptr(),
                                 ws.data_ptr(), nws, _stream_ptr(stream)), "exq_measure_exl2")
    return err


def exq_quantize_exl2(W, bits, perm=None, stream=None) -> Weight:
    """RTN conversion of an fp16 weight [K, N] (device) at the given widths
    [K/32] into an EXL2 layer."""
    import torch
    K, N = W.shape
    off = exq_exl2_seg_word_off(bits)
    rows = int(off[-1])
    off_d = torch.from_numpy(off.view(np.int32)).to(W.device)
    qw = torch.empty(rows, N, dtype=torch.int32, device=W.device)
    sc = torch.empty(K // 32, N, dtype=torch.float16, device=W.device)
    _check(_lib.exq_quantize_exl2(W.data_ptr(), None if perm is None else perm.data_ptr(), K, N, off_d.data_ptr(),
                                  rows, qw.data_ptr(), sc.data_ptr(), _stream_ptr(stream)), "exq_quantize_exl2")
    return Weight(EXQ_FMT_EXL2, K, N, 32, qw, sc, None, perm, off_d)


def exq_get_last_device_error(stream=None) -> int:
    return int(_lib.exq_get_last_device_error(_stream_ptr(stream)))


def exq_testing_starve(wait_rounds: int) -> None:
    """Failure-detection test hook (include/exq_testing.h): while wait_rounds
    > 0, GEMV / GEMM launches issue no copies and their bounded waits give up
    after wait_rounds rounds, so the call ends in EXQ_ERR_TIMEOUT; 0 = off."""
    _lib.exq_testing_starve(int(wait_rounds))
