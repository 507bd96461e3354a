"""ctypes binding of ``libw4a8.so`` (the C ABI in ``include/w4a8.h``).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels.  PyTorch supplies device memory and the current stream.  There is no CPU
fallback: if the library is missing or the GPU is not an sm_103 part, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libw4a8.so")

W4A8_OK = 0
W4A8_ERR_ARG = -1
W4A8_ERR_ALIGN = -2
W4A8_ERR_SHAPE = -3
W4A8_ERR_CUDA = -4
W4A8_ERR_TIMEOUT = -5
W4A8_ERR_WORKSPACE = -6
W4A8_ERR_DEVICE = -7
W4A8_ERR_SCRATCH_LIMIT = -8
NOALLOC_SCRATCH_BYTES = 16 << 20
OUT_F32 = 0
OUT_BF16 = 1
_OUT_DTYPES = {torch.float32: OUT_F32, torch.bfloat16: OUT_BF16}

# name -> (restype, argtypes); every symbol include/w4a8.h declares
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
SIGNATURES = {
    "w4a8_quant_pack": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P, _P]),
    "w4a8_linear": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "w4a8_prefill_linear": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "w4a8_prefill_linear_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w4a8_prepare_activations": (ctypes.c_int, [_P, _I64, _I64, _P, _SZ, _P]),
    "w4a8_prepare_weights": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _P, _SZ, _P]),
    "w4a8_linear_prepared": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w4a8_prefill_linear_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                              _I64, _I64, _I64, _P, _SZ, _P]),
    "w4a8_linear_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                      _I64, _I64, _I64, _P, _SZ, _P]),
    "w4a8_linear_prepared_ex": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                               _I64, _I64, _I64, _P]),
    "w4a8_prepared_activations_bytes": (_SZ, [_I64, _I64]),
    "w4a8_prepared_weights_bytes": (_SZ, [_I64, _I64]),
    "w4a8_linear_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "w4a8_prefill_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "w4a8_debug_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "w4a8_debug_block_acc": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I64, _I64, _I64, _I64, _P, _P, _SZ, _P]),
    "w4a8_tape_begin": (ctypes.c_int, [_P]),
    "w4a8_tape_end": (ctypes.c_int, [_P, ctypes.POINTER(_P)]),
    "w4a8_tape_replay": (ctypes.c_int, [_P, _P]),
    "w4a8_tape_free": (None, [_P]),
    "w4a8_sync_status": (ctypes.c_int, [_P]),
    "w4a8_selftest_wait_timeout": (ctypes.c_int, [_I64, _P]),
    "w4a8_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "w4a8_abi_version": (ctypes.c_int, []),
}

_lib = None


class W4A8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libw4a8.so not found at {path}: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().w4a8_status_string(int(status)).decode()


def _check(rc: int, where: str) -> None:
    if rc != W4A8_OK:
        raise W4A8Error(rc, where)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _want(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4a8_linear_workspace_bytes(M, N, K))


def prefill_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4a8_prefill_workspace_bytes(M, N, K))


def debug_workspace_bytes(m_cnt: int, n_cnt: int, K: int) -> int:
    return int(load().w4a8_debug_workspace_bytes(m_cnt, n_cnt, K))


def workspace(nbytes: int, device) -> torch.Tensor:
    """A caller-owned workspace buffer (uint8, at least 16-byte aligned)."""
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def quant_pack(x: torch.Tensor, a_q=None, a_scale=None, rowsum=None, stream=None):
    """w4a8_quant_pack: x fp32 [M,K] -> (a_q int8 [M,K], s_a fp32 [M], rowsum int32 [M,K/64])."""
    _want(x, torch.float32, "x")
    M, K = x.shape
    dev = x.device
    a_q = torch.empty((M, K), dtype=torch.int8, device=dev) if a_q is None else a_q
    a_scale = torch.empty((M,), dtype=torch.float32, device=dev) if a_scale is None else a_scale
    rowsum = torch.empty((M, K // 64), dtype=torch.int32, device=dev) if rowsum is None else rowsum
    rc = load().w4a8_quant_pack(_ptr(x), M, K, _ptr(a_q), _ptr(a_scale), _ptr(rowsum), _stream(stream))
    _check(rc, "w4a8_quant_pack")
    return a_q, a_scale, rowsum


def linear(a_q, a_scale, rowsum, wq, w_scale, w_zero, bias=None, y=None, ws=None, stream=None):
    """w4a8_linear: pre-quantized activations -> y fp32 [M,N]."""
    _want(a_q, torch.int8, "a_q")
    _want(wq, torch.uint8, "wq")
    _want(w_scale, torch.float16, "w_scale")
    _want(w_zero, torch.float16, "w_zero")
    M, K = a_q.shape
    N = wq.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=a_q.device) if y is None else y
    if ws is None:
        ws = workspace(linear_workspace_bytes(M, N, K), a_q.device)
    rc = load().w4a8_linear(_ptr(a_q), _ptr(a_scale), _ptr(rowsum), _ptr(wq), _ptr(w_scale), _ptr(w_zero),
                            _ptr(bias), _ptr(y), M, N, K, _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "w4a8_linear")
    return y


def prefill_linear(x, wq, w_scale, w_zero, bias=None, y=None, ws=None, stream=None):
    """w4a8_prefill_linear: fp32 x [M,K] -> y fp32 [M,N] (pre-pass + linear)."""
    _want(x, torch.float32, "x")
    _want(wq, torch.uint8, "wq")
    M, K = x.shape
    N = wq.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if y is None else y
    if ws is None:
        ws = workspace(prefill_workspace_bytes(M, N, K), x.device)
    rc = load().w4a8_prefill_linear(_ptr(x), _ptr(wq), _ptr(w_scale), _ptr(w_zero), _ptr(bias), _ptr(y),
                                    M, N, K, _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "w4a8_prefill_linear")
    return y


def prefill_linear_noalloc(x, wq, w_scale, w_zero, bias=None, y=None, stream=None):
    """w4a8_prefill_linear_noalloc: the fused call on the library's static scratch buffer,
    for callers that cannot allocate device memory.  Serialize calls that could overlap."""
    _want(x, torch.float32, "x")
    _want(wq, torch.uint8, "wq")
    M, K = x.shape
    N = wq.shape[0]
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if y is None else y
    rc = load().w4a8_prefill_linear_noalloc(_ptr(x), _ptr(wq), _ptr(w_scale), _ptr(w_zero), _ptr(bias), _ptr(y),
                                            M, N, K, _stream(stream))
    _check(rc, "w4a8_prefill_linear_noalloc")
    return y


def prepared_activations_bytes(M: int, K: int) -> int:
    return int(load().w4a8_prepared_activations_bytes(M, K))


def prepared_weights_bytes(N: int, K: int) -> int:
    return int(load().w4a8_prepared_weights_bytes(N, K))


def prepare_activations(x, act=None, stream=None):
    """w4a8_prepare_activations: the pre-pass into an opaque buffer (returned)."""
    _want(x, torch.float32, "x")
    M, K = x.shape
    act = workspace(prepared_activations_bytes(M, K), x.device) if act is None else act
    rc = load().w4a8_prepare_activations(_ptr(x), M, K, _ptr(act), act.numel(), _stream(stream))
    _check(rc, "w4a8_prepare_activations")
    return act


def prepare_weights(wq, w_scale, w_zero, pw=None, stream=None):
    """w4a8_prepare_weights: the tensor-core weight operand and the scale / zero layout
    (an opaque buffer, returned)."""
    _want(wq, torch.uint8, "wq")
    _want(w_scale, torch.float16, "w_scale")
    _want(w_zero, torch.float16, "w_zero")
    N, K = wq.shape[0], 2 * wq.shape[1]
    pw = workspace(prepared_weights_bytes(N, K), wq.device) if pw is None else pw
    rc = load().w4a8_prepare_weights(_ptr(wq), _ptr(w_scale), _ptr(w_zero), N, K, _ptr(pw), pw.numel(),
                                     _stream(stream))
    _check(rc, "w4a8_prepare_weights")
    return pw


def _out(y, shape, device, out_dtype):
    dt = torch.float32 if out_dtype is None else out_dtype
    if dt not in _OUT_DTYPES:
        raise TypeError(f"y: unsupported output dtype {dt}")
    y = torch.empty(shape, dtype=dt, device=device) if y is None else y
    if y.dtype != dt or not y.is_contiguous() or tuple(y.shape) != tuple(shape):
        raise ValueError(f"y: want a contiguous {dt} tensor of shape {tuple(shape)}")
    return y, _OUT_DTYPES[dt]


def prefill_linear_ex(x, wq, w_scale, w_zero, bias=None, y=None, out_dtype=None, clamp=(-math.inf, math.inf),
                      ws=None, stream=None):
    """w4a8_prefill_linear_ex: the fused call with the epilogue clamp and an fp32 or bf16 y."""
    _want(x, torch.float32, "x")
    _want(wq, torch.uint8, "wq")
    M, K = x.shape
    N = wq.shape[0]
    y, code = _out(y, (M, N), x.device, out_dtype if y is None else y.dtype)
    if ws is None:
        ws = workspace(prefill_workspace_bytes(M, N, K), x.device)
    rc = load().w4a8_prefill_linear_ex(_ptr(x), _ptr(wq), _ptr(w_scale), _ptr(w_zero), _ptr(bias), _ptr(y), code,
                                       float(clamp[0]), float(clamp[1]), M, N, K, _ptr(ws), ws.numel(),
                                       _stream(stream))
    _check(rc, "w4a8_prefill_linear_ex")
    return y


def linear_ex(a_q, a_scale, rowsum, wq, w_scale, w_zero, bias=None, y=None, out_dtype=None,
              clamp=(-math.inf, math.inf), ws=None, stream=None):
    """w4a8_linear_ex: pre-quantized activations, epilogue clamp, fp32 or bf16 y."""
    _want(a_q, torch.int8, "a_q")
    _want(wq, torch.uint8, "wq")
    M, K = a_q.shape
    N = wq.shape[0]
    y, code = _out(y, (M, N), a_q.device, out_dtype if y is None else y.dtype)
    if ws is None:
        ws = workspace(linear_workspace_bytes(M, N, K), a_q.device)
    rc = load().w4a8_linear_ex(_ptr(a_q), _ptr(a_scale), _ptr(rowsum), _ptr(wq), _ptr(w_scale), _ptr(w_zero),
                               _ptr(bias), _ptr(y), code, float(clamp[0]), float(clamp[1]), M, N, K, _ptr(ws),
                               ws.numel(), _stream(stream))
    _check(rc, "w4a8_linear_ex")
    return y


def linear_prepared_ex(act, pw, M: int, N: int, K: int, bias=None, y=None, out_dtype=None,
                       clamp=(-math.inf, math.inf), stream=None):
    """w4a8_linear_prepared_ex: prepared operands, epilogue clamp, fp32 or bf16 y."""
    y, code = _out(y, (M, N), act.device, out_dtype if y is None else y.dtype)
    rc = load().w4a8_linear_prepared_ex(_ptr(act), _ptr(pw), _ptr(bias), _ptr(y), code, float(clamp[0]),
                                        float(clamp[1]), M, N, K, _stream(stream))
    _check(rc, "w4a8_linear_prepared_ex")
    return y


def linear_prepared(act, pw, M: int, N: int, K: int, bias=None, y=None, stream=None):
    """w4a8_linear_prepared: contraction + epilogue from prepared operands -> y fp32 [M,N]."""
    y = torch.empty((M, N), dtype=torch.float32, device=act.device) if y is None else y
    rc = load().w4a8_linear_prepared(_ptr(act), _ptr(pw), _ptr(bias), _ptr(y), M, N, K, _stream(stream))
    _check(rc, "w4a8_linear_prepared")
    return y


def debug_block_acc(a_q, wq, N, m0=0, m_cnt=None, n0=0, n_cnt=None, ws=None, stream=None):
    """w4a8_debug_block_acc: exact per-block int32 accumulators [m_cnt, n_cnt, K/64]."""
    _want(a_q, torch.int8, "a_q")
    M, K = a_q.shape
    m_cnt = M - m0 if m_cnt is None else m_cnt
    n_cnt = N - n0 if n_cnt is None else n_cnt
    acc = torch.empty((m_cnt, n_cnt, K // 64), dtype=torch.int32, device=a_q.device)
    if ws is None:
        ws = workspace(debug_workspace_bytes(m_cnt, n_cnt, K), a_q.device)
    rc = load().w4a8_debug_block_acc(_ptr(a_q), _ptr(wq), M, N, K, m0, m_cnt, n0, n_cnt, _ptr(acc),
                                     _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "w4a8_debug_block_acc")
    return acc


def sync_status(stream=None) -> int:
    """Synchronize the stream and return (and clear) the device status word."""
    return int(load().w4a8_sync_status(_stream(stream)))


def selftest_wait_timeout(limit_us: int, stream=None) -> None:
    _check(load().w4a8_selftest_wait_timeout(int(limit_us), _stream(stream)), "w4a8_selftest_wait_timeout")


class Tape:
    """A recorded call sequence (w4a8_tape_*): `with Tape(stream) as t:` records the library
    calls made on `stream` inside the block; `t.replay(stream)` runs them again with one
    launch.  The tensors the recorded calls used must stay alive while the tape is."""

    def __init__(self, stream):
        self.stream = stream
        self.handle = None

    def __enter__(self):
        _check(load().w4a8_tape_begin(_stream(self.stream)), "w4a8_tape_begin")
        return self

    def __exit__(self, exc_type, exc, tb):
        h = _P()
        rc = load().w4a8_tape_end(_stream(self.stream), ctypes.byref(h))
        if exc_type is None:
            _check(rc, "w4a8_tape_end")
            self.handle = h
        elif rc == 0 and h:
            load().w4a8_tape_free(h)
        return False

    def replay(self, stream=None):
        if self.handle is None:
            raise RuntimeError("tape not recorded")
        _check(load().w4a8_tape_replay(self.handle, _stream(stream)), "w4a8_tape_replay")

    def free(self):
        if self.handle is not None:
            load().w4a8_tape_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

