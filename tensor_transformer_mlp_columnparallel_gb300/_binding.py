"""ctypes binding of libtpmlp.so (include/tpmlp.h).

Argument marshalling only: tensors become device pointers, lists of shard
tensors become host arrays of pointers, the current torch stream becomes the
cudaStream_t. Every step of the computation runs in the library's CUDA
kernels; there is no fallback. If the shared library is missing, loading
raises instead of silently doing something else.
"""

import ctypes
import os
import re
from typing import List, Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtpmlp.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "tpmlp.h")

MAX_SHARDS = 16
OK, ERR_ARG, ERR_SHAPE, ERR_ALIGN, ERR_DTYPE, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(8)
ACT = {"relu": 0, "gelu_tanh": 1, "gelu_erf": 2, "gelu_sigmoid": 3}
DTYPE = {torch.float32: 0, torch.bfloat16: 1}
MODE = {"partials": 0, "splitk": 1}
OP_FORWARD, OP_BACKWARD = 0, 1


class TpmlpError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


class KernelTiming(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 48), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_PP = ctypes.POINTER(ctypes.c_void_p)

_SIGNATURES = {
    "tpmlp_forward": (_int, [_int, _i64, _i64, _i64, _int, _int, _vp, _PP, _PP, _PP, _vp, _vp,
                             _PP, _PP, _int, _vp, ctypes.c_size_t, _vp]),
    "tpmlp_forward_noalloc": (_int, [_int, _i64, _i64, _i64, _int, _int, _vp, _PP, _PP, _PP, _vp,
                                     _vp, _PP, _PP, _vp]),
    "tpmlp_swiglu_forward": (_int, [_int, _i64, _i64, _i64, _int, _vp, _PP, _PP, _PP, _vp, _PP, _PP,
                                    _PP, _int, _vp, ctypes.c_size_t, _vp]),
    "tpmlp_backward": (_int, [_int, _i64, _i64, _i64, _int, _int, _vp, _PP, _PP, _PP, _PP, _vp,
                              _vp, _PP, _PP, _PP, _vp, _int, _vp, ctypes.c_size_t, _vp]),
    "tpmlp_block_reduce": (_int, [_int, _i64, _i64, _int, _PP, _vp, _vp, _vp]),
    "tpmlp_block_reduce_scatter": (_int, [_int, _i64, _i64, _int, _PP, _vp, _PP, _vp]),
    "tpmlp_forward_reduce_scatter": (_int, [_int, _i64, _i64, _i64, _int, _int, _vp, _PP, _PP, _PP,
                                            _vp, _PP, _PP, _PP, _int, _vp, ctypes.c_size_t, _vp]),
    "tpmlp_vocab_embedding": (_int, [_int, _i64, _i64, _i64, _int, _vp, _PP, _vp, _vp]),
    "tpmlp_vocab_ce": (_int, [_i64, _i64, _int, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "tpmlp_vocab_ce_backward": (_int, [_i64, _i64, _int, _vp, _vp, _vp, ctypes.c_float, _vp, _vp]),
    "tpmlp_workspace_bytes": (ctypes.c_size_t, [_int, _int, _i64, _i64, _i64, _int, _int]),
    "tpmlp_workspace_bytes_balanced": (ctypes.c_size_t, [_int, _int, _i64, _i64, _i64, _int, _int]),
    "tpmlp_status_str": (ctypes.c_char_p, [_int]),
    "tpmlp_check_device_error": (_int, [_vp]),
    "tpmlp_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
    "tpmlp_selftest_wait_timeout": (_int, [ctypes.c_uint64, _vp]),
    "tpmlp_selftest_gemm_stall": (_int, [_int]),
    "tpmlp_launch_count": (ctypes.c_int64, []),
    "tpmlp_gemm_plan": (_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _int, _int, _int,
                               _int, ctypes.POINTER(_int), ctypes.POINTER(_int),
                               ctypes.POINTER(_int)]),
    "tpmlp_timing_enable": (None, [_int]),
    "tpmlp_timing_read": (_int, [ctypes.POINTER(KernelTiming), _int]),
    "tpmlp_timing_reset": (None, []),
}


def lib():
    """The loaded library (loads it on first use; raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def header_functions() -> List[str]:
    """Names of the functions include/tpmlp.h declares."""
    src = open(HEADER_PATH).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tpmlp_[a-z_]+)\s*\(", src)))


def status_str(status: int) -> str:
    return lib().tpmlp_status_str(int(status)).decode()


def _check(status: int):
    if status != OK:
        raise TpmlpError(status, status_str(status))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _ptrs(ts: Optional[Sequence[torch.Tensor]]):
    if ts is None:
        return None
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = t.data_ptr()
    return ctypes.cast(arr, _PP)


def _stream(t: torch.Tensor):
    if t.is_cuda:
        return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)
    return None


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in DTYPE:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return DTYPE[t.dtype]


def _require(ts, device, dtype):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or t.device != device:
            raise ValueError("all tensors must live on the same CUDA device")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"expected {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous (row-major)")


# ---------------------------------------------------------------------------
# The C-ABI calls, same names, tensors in place of pointers
# ---------------------------------------------------------------------------

def tpmlp_workspace_bytes(op: int, dtype: torch.dtype, N: int, D: int, F: int, T: int,
                          mode: str) -> int:
    return int(lib().tpmlp_workspace_bytes(op, DTYPE[dtype], N, D, F, T, MODE[mode]))


def tpmlp_workspace_bytes_balanced(op: int, dtype: torch.dtype, N: int, D: int, F: int, T: int,
                                   mode: str) -> int:
    """Workspace size that also holds the few-token GEMMs' stream-K scratch
    (see include/tpmlp.h)."""
    return int(lib().tpmlp_workspace_bytes_balanced(op, DTYPE[dtype], N, D, F, T, MODE[mode]))


def tpmlp_forward(X, W1, b1, W2, b2, Y, H, Z, act: str, mode: str, workspace=None):
    """Y = sum_r act(X W1[r] + b1[r]) W2[r] + b2 (see include/tpmlp.h).
    W1, W2, H, Z, b1 are lists of T tensors (b1, Z may be None)."""
    T = len(W1)
    N, D = X.shape
    Fs = W1[0].shape[1]
    _require([X, b2, Y, *W1, *W2, *H, *(b1 or []), *(Z or [])], X.device, X.dtype)
    _require([workspace], X.device, None)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().tpmlp_forward(_dtype_code(X), N, D, Fs * T, T, ACT[act], _ptr(X), _ptrs(W1),
                               _ptrs(b1), _ptrs(W2), _ptr(b2), _ptr(Y), _ptrs(H), _ptrs(Z),
                               MODE[mode], _ptr(workspace), ws_bytes, _stream(X)))


def tpmlp_forward_noalloc(X, W1, b1, W2, b2, Y, H, Z, act: str):
    """tpmlp_forward in PARTIALS mode with the partial sums in the library's
    own fixed scratch array (no workspace, no device allocation); see
    include/tpmlp.h for its size limit and the sharing rules."""
    T = len(W1)
    N, D = X.shape
    Fs = W1[0].shape[1]
    _require([X, b2, Y, *W1, *W2, *H, *(b1 or []), *(Z or [])], X.device, X.dtype)
    _check(lib().tpmlp_forward_noalloc(_dtype_code(X), N, D, Fs * T, T, ACT[act], _ptr(X),
                                       _ptrs(W1), _ptrs(b1), _ptrs(W2), _ptr(b2), _ptr(Y),
                                       _ptrs(H), _ptrs(Z), _stream(X)))


def tpmlp_swiglu_forward(X, Wg, Wu, Wd, Y, H, G, U, mode: str, workspace=None):
    """Gated block: H^(r) = SiLU(X Wg[r]) * (X Wu[r]), Y = sum_r H^(r) Wd[r]."""
    T = len(Wg)
    N, D = X.shape
    Fs = Wg[0].shape[1]
    _require([X, Y, *Wg, *Wu, *Wd, *H, *(G or []), *(U or [])], X.device, X.dtype)
    _require([workspace], X.device, None)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().tpmlp_swiglu_forward(_dtype_code(X), N, D, Fs * T, T, _ptr(X), _ptrs(Wg),
                                      _ptrs(Wu), _ptrs(Wd), _ptr(Y), _ptrs(H), _ptrs(G), _ptrs(U),
                                      MODE[mode], _ptr(workspace), ws_bytes, _stream(X)))


def tpmlp_backward(X, W1, W2, H, Z, dY, dX, dW1, dW2, db1, db2, act: str, mode: str, workspace):
    """Gradients of the block for upstream dY (see include/tpmlp.h)."""
    T = len(W1)
    N, D = X.shape
    Fs = W1[0].shape[1]
    _require([X, dY, dX, db2, *W1, *W2, *H, *Z, *dW1, *dW2, *(db1 or [])], X.device, X.dtype)
    _require([workspace], X.device, None)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().tpmlp_backward(_dtype_code(X), N, D, Fs * T, T, ACT[act], _ptr(X), _ptrs(W1),
                                _ptrs(W2), _ptrs(H), _ptrs(Z), _ptr(dY), _ptr(dX), _ptrs(dW1),
                                _ptrs(dW2), _ptrs(db1), _ptr(db2), MODE[mode], _ptr(workspace),
                                ws_bytes, _stream(X)))


def tpmlp_block_reduce(partials: Sequence[torch.Tensor], b2, Y):
    """Y = sum_r partials[r] + b2, fp32 partials, Y fp32 or bf16."""
    T = len(partials)
    N, D = Y.shape
    _require([*partials], Y.device, torch.float32)
    _require([b2, Y], Y.device, Y.dtype)
    for p in partials:
        if p.dtype != torch.float32:
            raise TypeError("partial sums are fp32")
    _check(lib().tpmlp_block_reduce(_dtype_code(Y), N, D, T, _ptrs(partials), _ptr(b2), _ptr(Y),
                                    _stream(Y)))


def tpmlp_block_reduce_scatter(partials: Sequence[torch.Tensor], b2, Y_rows: Sequence[torch.Tensor]):
    """Rows [r N/T, (r+1) N/T) of sum_r partials[r] + b2 into Y_rows[r]."""
    T = len(partials)
    N, D = partials[0].shape
    _require([*partials], partials[0].device, torch.float32)
    _require([b2, *Y_rows], partials[0].device, Y_rows[0].dtype)
    _check(lib().tpmlp_block_reduce_scatter(_dtype_code(Y_rows[0]), N, D, T, _ptrs(partials),
                                            _ptr(b2), _ptrs(Y_rows), _stream(partials[0])))


def tpmlp_forward_reduce_scatter(X, W1, b1, W2, b2, Y_rows, H, Z, act: str, mode: str,
                                 workspace=None):
    """tpmlp_forward with the reduce-scatter block end: rank r's rows in Y_rows[r]."""
    T = len(W1)
    N, D = X.shape
    Fs = W1[0].shape[1]
    _require([X, b2, *Y_rows, *W1, *W2, *H, *(b1 or []), *(Z or [])], X.device, X.dtype)
    _require([workspace], X.device, None)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().tpmlp_forward_reduce_scatter(
        _dtype_code(X), N, D, Fs * T, T, ACT[act], _ptr(X), _ptrs(W1), _ptrs(b1), _ptrs(W2),
        _ptr(b2), _ptrs(Y_rows), _ptrs(H), _ptrs(Z), MODE[mode], _ptr(workspace), ws_bytes,
        _stream(X)))


def tpmlp_vocab_embedding(ids, table: Sequence[torch.Tensor], out):
    """out[n] = table row ids[n] (table split by rows into len(table) shards)."""
    T = len(table)
    Vs, Hd = table[0].shape
    _require([ids], out.device, torch.int64)
    _require([*table, out], out.device, out.dtype)
    _check(lib().tpmlp_vocab_embedding(_dtype_code(out), ids.shape[0], Vs * T, Hd, T, _ptr(ids),
                                       _ptrs(table), _ptr(out), _stream(out)))


def tpmlp_vocab_ce(logits, targets, T: int, loss_per_token, loss_mean=None, argmax=None,
                   target_owner=None):
    """Vocab-parallel cross-entropy over T contiguous vocab shards."""
    N, V = logits.shape
    _require([logits], logits.device, torch.float32)
    _require([targets], logits.device, torch.int64)
    _require([loss_per_token, loss_mean], logits.device, torch.float32)
    _require([argmax, target_owner], logits.device, torch.int32)
    _check(lib().tpmlp_vocab_ce(N, V, T, _ptr(logits), _ptr(targets), _ptr(loss_per_token),
                                _ptr(loss_mean), _ptr(argmax), _ptr(target_owner),
                                _stream(logits)))


def tpmlp_vocab_ce_backward(logits, targets, T: int, loss_per_token, grad_scale: float, dlogits):
    """dlogits = grad_scale * (softmax(logits) - onehot(targets)); dlogits may
    be logits itself (in place)."""
    N, V = logits.shape
    _require([logits, loss_per_token, dlogits], logits.device, torch.float32)
    _require([targets], logits.device, torch.int64)
    _check(lib().tpmlp_vocab_ce_backward(N, V, T, _ptr(logits), _ptr(targets), _ptr(loss_per_token),
                                         float(grad_scale), _ptr(dlogits), _stream(logits)))


def tpmlp_check_device_error(device=None) -> int:
    """Synchronizes the current stream and returns (and clears) the device
    error word: OK, ERR_TIMEOUT or ERR_ARG."""
    s = torch.cuda.current_stream(device).cuda_stream
    return int(lib().tpmlp_check_device_error(ctypes.c_void_p(s)))


def tpmlp_set_wait_timeout_ns(ns: int):
    lib().tpmlp_set_wait_timeout_ns(int(ns))


def tpmlp_selftest_wait_timeout(timeout_ns: int, device=None):
    s = torch.cuda.current_stream(device).cuda_stream
    _check(lib().tpmlp_selftest_wait_timeout(int(timeout_ns), ctypes.c_void_p(s)))


def tpmlp_selftest_gemm_stall(role: int):
    """While role is 1 (epilogue), 2 (MMA issuer) or 3 (TMA producer), every
    bf16 GEMM launch makes that role stall on a barrier nothing completes
    until the bounded wait runs out; 0 turns it off."""
    _check(lib().tpmlp_selftest_gemm_stall(int(role)))


def tpmlp_launch_count() -> int:
    return int(lib().tpmlp_launch_count())


def tpmlp_gemm_plan(M: int, N: int, K: int, G: int, fold: bool = False, dual: bool = False,
                    balanced: bool = False):
    """Launch configuration of the bf16 tensor-core GEMM for this shape on the
    current device: (accumulator columns, CTAs per MMA, K split: cluster size,
    or 0 for stream-K, which needs balanced=True)."""
    bn, ctas, ks = _int(0), _int(0), _int(0)
    _check(lib().tpmlp_gemm_plan(M, N, K, G, 1 if fold else 0, 1 if dual else 0,
                                 1 if balanced else 0, ctypes.byref(bn), ctypes.byref(ctas),
                                 ctypes.byref(ks)))
    return bn.value, ctas.value, ks.value


def tpmlp_timing_enable(on: bool):
    lib().tpmlp_timing_enable(1 if on else 0)


def tpmlp_timing_read() -> dict:
    buf = (KernelTiming * 64)()
    n = lib().tpmlp_timing_read(buf, 64)
    if n < 0:
        raise TpmlpError(ERR_CUDA, "timing read failed")
    return {buf[i].name.decode(): {"launches": int(buf[i].launches), "total_ms": float(buf[i].total_ms)}
            for i in range(n)}


def tpmlp_timing_reset():
    lib().tpmlp_timing_reset()
