"""Thin ctypes binding over libbitmtp_linear.so (include/bitmtp_linear.h).

Argument marshalling only: every step of the linear runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  The raw
entry points keep the C names (``bitmtp_linear_*``); ``pack``,
``ternarize_pack``, ``quant_act``, ``gemm`` and ``gemm_grouped`` are tensor
conveniences over them.

The library must have been built (``ternary_w2a8_linear_gb300.build``); if it
is missing this module raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbitmtp_linear.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "bitmtp_linear.h")

OK = 0
ERR_INVALID, ERR_ALIGN, ERR_SHAPE, ERR_NOT_TERNARY, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE, ERR_NOT_FINITE = \
    range(-1, -9, -1)
F32, BF16, Q8 = 0, 1, 2
FLAG_PDL, FLAG_FORCE_TC, FLAG_FORCE_DP, FLAG_TEST_WITHHOLD = 0x1, 0x2, 0x4, 0x100
FLAG_FP8 = 0x8  # "fast" draft projection: FP8 (E4M3) activations; acc holds fp32 bit patterns
MAX_M, MAX_K, MAX_N, MAX_GROUP = 16, 32768, 16777216, 8
NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024


class BitmtpError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what else status_string(status))


class Act(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("x", ctypes.c_void_p), ("ldx", ctypes.c_int64),
                ("a_scale", ctypes.c_void_p), ("amax", ctypes.c_void_p)]


class Out(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("y", ctypes.c_void_p), ("ldy", ctypes.c_int64),
                ("acc", ctypes.c_void_p), ("lda", ctypes.c_int64), ("amax", ctypes.c_void_p)]


class TernDesc(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("ldw", ctypes.c_int64),
                ("pk", ctypes.c_void_p), ("pk_bytes", ctypes.c_size_t), ("w_scale", ctypes.c_void_p)]


class GemmDesc(ctypes.Structure):
    _fields_ = [("pk", ctypes.c_void_p), ("w_scale", ctypes.c_float), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("M", ctypes.c_int64), ("act", Act), ("out", Out)]


_lib = None


def load() -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m ternary_w2a8_linear_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    c = ctypes
    sig = {
        "bitmtp_linear_packed_bytes": (c.c_size_t, [c.c_int64, c.c_int64]),
        "bitmtp_linear_pack": (c.c_int, [c.c_void_p, c.c_int64, c.c_int64, c.c_int64, c.c_void_p,
                                         c.c_size_t, c.c_void_p]),
        "bitmtp_linear_ternarize_workspace_bytes": (c.c_size_t, [c.c_int64, c.c_int64]),
        "bitmtp_linear_ternarize_pack": (c.c_int, [c.c_void_p, c.c_int64, c.c_int64, c.c_int64, c.c_void_p,
                                                   c.c_size_t, c.c_void_p, c.c_void_p, c.c_size_t,
                                                   c.c_void_p]),
        "bitmtp_linear_ternarize_workspace_bytes_grouped": (c.c_size_t, [c.c_int]),
        "bitmtp_linear_ternarize_pack_grouped": (c.c_int, [c.POINTER(TernDesc), c.c_int, c.c_void_p, c.c_size_t,
                                                           c.c_void_p]),
        "bitmtp_linear_quant_act": (c.c_int, [c.c_void_p, c.c_int, c.c_int64, c.c_int64, c.c_int64,
                                              c.c_void_p, c.c_int64, c.c_void_p, c.c_void_p, c.c_void_p]),
        "bitmtp_linear_workspace_bytes": (c.c_size_t, [c.c_int64, c.c_int64, c.c_int64]),
        "bitmtp_linear_workspace_bytes_grouped": (c.c_size_t, [c.POINTER(GemmDesc), c.c_int]),
        "bitmtp_linear_gemm": (c.c_int, [c.c_void_p, c.c_float, c.c_int64, c.c_int64, c.c_int64,
                                         c.POINTER(Act), c.POINTER(Out), c.c_void_p, c.c_size_t,
                                         c.c_uint, c.c_void_p]),
        "bitmtp_linear_gemm_grouped": (c.c_int, [c.POINTER(GemmDesc), c.c_int, c.c_void_p, c.c_size_t,
                                                 c.c_uint, c.c_void_p]),
        "bitmtp_linear_gemm_noalloc": (c.c_int, [c.c_void_p, c.c_float, c.c_int64, c.c_int64, c.c_int64,
                                                 c.POINTER(Act), c.POINTER(Out), c.c_uint, c.c_void_p]),
        "bitmtp_linear_device_error": (c.c_int, [c.c_void_p]),
        "bitmtp_linear_status_string": (c.c_char_p, [c.c_int]),
        "bitmtp_linear_version": (c.c_int, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def header_symbols() -> list[str]:
    """Every function the public header declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(bitmtp_linear_\w+)\s*\(", text, re.M)))


# ---------------------------------------------------------------- raw ABI --
def bitmtp_linear_packed_bytes(N: int, K: int) -> int:
    return int(load().bitmtp_linear_packed_bytes(N, K))


def bitmtp_linear_pack(T_ptr, N, K, ldt, pk_ptr, pk_bytes, stream) -> int:
    return load().bitmtp_linear_pack(T_ptr, N, K, ldt, pk_ptr, pk_bytes, stream)


def bitmtp_linear_ternarize_workspace_bytes(N: int, K: int) -> int:
    return int(load().bitmtp_linear_ternarize_workspace_bytes(N, K))


def bitmtp_linear_ternarize_pack(W_ptr, N, K, ldw, pk_ptr, pk_bytes, w_scale_ptr, ws_ptr, ws_bytes, stream) -> int:
    return load().bitmtp_linear_ternarize_pack(W_ptr, N, K, ldw, pk_ptr, pk_bytes, w_scale_ptr, ws_ptr, ws_bytes,
                                               stream)


def bitmtp_linear_quant_act(x_ptr, x_kind, M, K, ldx, q_ptr, ldq, a_scale_ptr, rowsum_ptr, stream) -> int:
    return load().bitmtp_linear_quant_act(x_ptr, x_kind, M, K, ldx, q_ptr, ldq, a_scale_ptr, rowsum_ptr, stream)


def bitmtp_linear_workspace_bytes(N: int, K: int, M: int) -> int:
    return int(load().bitmtp_linear_workspace_bytes(N, K, M))


def bitmtp_linear_workspace_bytes_grouped(descs) -> int:
    arr = (GemmDesc * max(1, len(descs)))(*descs)
    return int(load().bitmtp_linear_workspace_bytes_grouped(arr, len(descs)))


def bitmtp_linear_gemm(pk_ptr, w_scale, N, K, M, act: Act, out: Out, ws_ptr, ws_bytes, flags, stream) -> int:
    return load().bitmtp_linear_gemm(pk_ptr, w_scale, N, K, M, ctypes.byref(act), ctypes.byref(out),
                                     ws_ptr, ws_bytes, flags, stream)


def bitmtp_linear_gemm_grouped(descs, ws_ptr, ws_bytes, flags, stream) -> int:
    arr = (GemmDesc * max(1, len(descs)))(*descs)
    return load().bitmtp_linear_gemm_grouped(arr, len(descs), ws_ptr, ws_bytes, flags, stream)


def bitmtp_linear_gemm_noalloc(pk_ptr, w_scale, N, K, M, act: Act, out: Out, flags, stream) -> int:
    """bitmtp_linear_gemm on the library's built-in scratch array (no workspace,
    nothing allocated); calls on one device must not overlap on the GPU."""
    return load().bitmtp_linear_gemm_noalloc(pk_ptr, w_scale, N, K, M, ctypes.byref(act), ctypes.byref(out),
                                             flags, stream)


def bitmtp_linear_device_error(stream=None) -> int:
    return load().bitmtp_linear_device_error(_stream(stream))


def bitmtp_linear_status_string(status: int) -> str:
    return load().bitmtp_linear_status_string(status).decode()


def bitmtp_linear_version() -> int:
    return load().bitmtp_linear_version()


status_string = bitmtp_linear_status_string


def _check(status: int, what: str):
    if status != OK:
        raise BitmtpError(status, what)


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _act_kind(x: torch.Tensor) -> int:
    if x.dtype == torch.float32:
        return F32
    if x.dtype == torch.bfloat16:
        return BF16
    if x.dtype == torch.int8:
        return Q8
    raise TypeError(f"unsupported activation dtype {x.dtype}")


def _rowmajor(t: torch.Tensor, name: str) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit stride along columns")
    return t.stride(0)


# ------------------------------------------------------- tensor wrappers --
def packed_bytes(N: int, K: int) -> int:
    return bitmtp_linear_packed_bytes(N, K)


_ws_cache: dict = {}


def workspace(nbytes: int, device=None, stream=None) -> torch.Tensor:
    """A workspace of at least ``nbytes`` for GEMM calls on ``stream`` (cached
    per device and stream; calls on one stream are ordered, so they may share
    it).  Zero-filled once on allocation, as the library requires."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    sptr = _stream(stream).value or 0
    key = (dev.index, sptr)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        size = max(nbytes, 2 * ws.numel() if ws is not None else 0, 1 << 20)
        ws = torch.zeros(size, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize(dev)  # zero-fill complete before any stream uses it
        _ws_cache[key] = ws
    return ws


def pack(T: torch.Tensor, stream=None) -> torch.Tensor:
    """Pack ternary int8 weights [N, K] (device) -> uint8 packed buffer."""
    if T.dtype != torch.int8 or not T.is_cuda:
        raise TypeError("T must be a CUDA int8 tensor")
    N, K = T.shape
    ldt = _rowmajor(T, "T")
    nb = packed_bytes(N, K)
    if nb == 0:
        raise BitmtpError(ERR_SHAPE, "pack")
    pk = torch.empty(nb, dtype=torch.uint8, device=T.device)
    _check(bitmtp_linear_pack(_ptr(T), N, K, ldt, _ptr(pk), nb, _stream(stream)), "pack")
    return pk


def ternarize_pack(W: torch.Tensor, stream=None):
    """Absmean-ternarise fp32 weights [N, K] (device) and pack them on the
    device -> (packed uint8 buffer, w_scale as a Python float).  The scratch is
    a fresh tensor, not the GEMM workspace (which must stay zero-filled)."""
    if W.dtype != torch.float32 or not W.is_cuda:
        raise TypeError("W must be a CUDA float32 tensor")
    N, K = W.shape
    ldw = _rowmajor(W, "W")
    nb = packed_bytes(N, K)
    wb = bitmtp_linear_ternarize_workspace_bytes(N, K)
    if nb == 0 or wb == 0:
        raise BitmtpError(ERR_SHAPE, "ternarize_pack")
    pk = torch.empty(nb, dtype=torch.uint8, device=W.device)
    ws = torch.empty(wb, dtype=torch.uint8, device=W.device)
    g = torch.empty(1, dtype=torch.float32, device=W.device)
    _check(bitmtp_linear_ternarize_pack(_ptr(W), N, K, ldw, _ptr(pk), nb, _ptr(g), _ptr(ws), wb, _stream(stream)),
           "ternarize_pack")
    return pk, float(g.item())


def bitmtp_linear_ternarize_workspace_bytes_grouped(n_desc: int) -> int:
    return int(load().bitmtp_linear_ternarize_workspace_bytes_grouped(n_desc))


def bitmtp_linear_ternarize_pack_grouped(descs, n_desc, ws_ptr, ws_bytes, stream) -> int:
    return load().bitmtp_linear_ternarize_pack_grouped(descs, n_desc, ws_ptr, ws_bytes, stream)


def ternarize_pack_grouped(Ws, stream=None):
    """ternarize_pack of several fp32 weight matrices in one grouped call
    (four launches, one sync) -> list of (packed uint8 buffer, w_scale)."""
    n = len(Ws)
    wb = bitmtp_linear_ternarize_workspace_bytes_grouped(n)
    if wb == 0:
        raise BitmtpError(ERR_INVALID, "ternarize_pack_grouped")
    outs, descs = [], []
    for W in Ws:
        if W.dtype != torch.float32 or not W.is_cuda:
            raise TypeError("W must be a CUDA float32 tensor")
        N, K = W.shape
        ldw = _rowmajor(W, "W")
        nb = packed_bytes(N, K)
        if nb == 0:
            raise BitmtpError(ERR_SHAPE, "ternarize_pack_grouped")
        pk = torch.empty(nb, dtype=torch.uint8, device=W.device)
        g = torch.empty(1, dtype=torch.float32, device=W.device)
        outs.append((pk, g))
        descs.append(TernDesc(_ptr(W), N, K, ldw, _ptr(pk), nb, _ptr(g)))
    ws = torch.empty(wb, dtype=torch.uint8, device=Ws[0].device)
    arr = (TernDesc * n)(*descs)
    _check(bitmtp_linear_ternarize_pack_grouped(arr, n, _ptr(ws), wb, _stream(stream)), "ternarize_pack_grouped")
    return [(pk, float(g.item())) for pk, g in outs]


def quant_act(x: torch.Tensor, stream=None):
    """Per-row absmax int8 quantisation -> (q int8 [M,K], a_scale fp32 [M], rowsum int32 [M])."""
    kind = _act_kind(x)
    if kind == Q8:
        raise TypeError("x must be float32 or bfloat16")
    M, K = x.shape
    ldx = _rowmajor(x, "x")
    q = torch.empty((M, K), dtype=torch.int8, device=x.device)
    a_scale = torch.empty(M, dtype=torch.float32, device=x.device)
    rowsum = torch.empty(M, dtype=torch.int32, device=x.device)
    _check(bitmtp_linear_quant_act(_ptr(x), kind, M, K, ldx, _ptr(q), K, _ptr(a_scale), _ptr(rowsum),
                                   _stream(stream)), "quant_act")
    return q, a_scale, rowsum


def make_act(x: torch.Tensor, a_scale: torch.Tensor | None = None, amax: torch.Tensor | None = None) -> Act:
    kind = _act_kind(x)
    if kind == Q8 and a_scale is None:
        raise ValueError("int8 activations need a_scale")
    return Act(kind, x.data_ptr(), _rowmajor(x, "x"), a_scale.data_ptr() if kind == Q8 else None,
               amax.data_ptr() if amax is not None else None)


def make_out(y: torch.Tensor, acc: torch.Tensor | None = None, amax: torch.Tensor | None = None) -> Out:
    dt = F32 if y.dtype == torch.float32 else BF16 if y.dtype == torch.bfloat16 else None
    if dt is None:
        raise TypeError("y must be float32 or bfloat16")
    return Out(dt, y.data_ptr(), _rowmajor(y, "y"),
               acc.data_ptr() if acc is not None else None,
               _rowmajor(acc, "acc") if acc is not None else 0,
               amax.data_ptr() if amax is not None else None)


def gemm(pk: torch.Tensor, w_scale: float, N: int, K: int, x: torch.Tensor,
         a_scale: torch.Tensor | None = None, out_dtype=torch.float32, y: torch.Tensor | None = None,
         acc: torch.Tensor | bool | None = None, flags: int = 0, stream=None,
         workspace_tensor: torch.Tensor | None = None):
    """y = W2A8 linear of x ([M, K] fp32 / bf16 raw, or int8 codes with a_scale).

    Returns y, or (y, acc) when ``acc`` is True or a tensor.  With FLAG_FP8
    the int32 acc tensor holds the fp32 accumulators' bit patterns
    (``acc.view(torch.float32)``)."""
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=out_dtype, device=x.device)
    want_acc = acc is not None and acc is not False
    if acc is True:
        acc = torch.empty((M, N), dtype=torch.int32, device=x.device)
    act = make_act(x, a_scale)
    out = make_out(y, acc if want_acc else None)
    nb = bitmtp_linear_workspace_bytes(N, K, max(M, 1))
    ws = workspace_tensor if workspace_tensor is not None else (workspace(nb, x.device, stream) if M else None)
    _check(bitmtp_linear_gemm(_ptr(pk), float(w_scale), N, K, M, act, out, _ptr(ws),
                              ws.numel() if ws is not None else 0, flags, _stream(stream)), "gemm")
    return (y, acc) if want_acc else y


def gemm_grouped(problems, flags: int = 0, stream=None, workspace_tensor: torch.Tensor | None = None):
    """One launch over several problems.  Each problem is a dict with keys
    pk, w_scale, N, K, x, (a_scale), (amax: the rows' absmax handed over),
    y, (acc), (amax_out: receives the output rows' absmax)."""
    descs = []
    for p in problems:
        x = p["x"]
        descs.append(GemmDesc(p["pk"].data_ptr(), float(p["w_scale"]), p["N"], p["K"], x.shape[0],
                              make_act(x, p.get("a_scale"), p.get("amax")),
                              make_out(p["y"], p.get("acc"), p.get("amax_out"))))
    if not descs:
        return
    nb = bitmtp_linear_workspace_bytes_grouped(descs)
    dev = problems[0]["x"].device
    ws = workspace_tensor if workspace_tensor is not None else workspace(nb, dev, stream)
    _check(bitmtp_linear_gemm_grouped(descs, _ptr(ws), ws.numel(), flags, _stream(stream)), "gemm_grouped")
