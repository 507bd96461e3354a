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
    "w4a8_prefill_linear_batch": (ctypes.c_int, [_P, _I64, _I64, _P]),
    "w4a8_prepare_activations": (ctypes.c_int, [_P, _I64, _I64, _P, _SZ, _P]),
    "w4a8_prepare_weights": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _P, _SZ, _P]),
    "w4a8_linear_prepared": (ctypes.c_int, [_P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w4a8_linear_act": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "w4a8_linear_act_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "w4a8_prefill_linear_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                              _I64, _I64, _I64, _P, _SZ, _P]),
    "w4a8_linear_ex": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                      _I64, _I64, _I64, _P, _SZ, _P]),
    "w4a8_linear_prepared_ex": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                               _I64, _I64, _I64, _P]),
    "w4a8_prefill_linear_host": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "w4a8_prefill_host_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
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
    "w4a8_tape_kernels": (ctypes.c_int64, [_P]),
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


def _arg(t, dtype, shape, name: str, device=None, min_bytes=None):
    """Check one tensor argument before its address reaches the library, which cannot: a CUDA
    tensor on the call's device, contiguous, of the dtype and shape the C layout fixes (or, for
    an opaque buffer, at least ``min_bytes`` long).  ``None`` passes (optional arguments)."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (the library has no CPU path), got {t.device}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call's other tensors on {device}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if min_bytes is not None and _nbytes(t) < min_bytes:
        raise ValueError(f"{name} holds {_nbytes(t)} bytes, the call needs {min_bytes}")


def _want(t: torch.Tensor, dtype, name: str):
    _arg(t, dtype, None, name)
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device} but the current CUDA device is "
                         f"{torch.cuda.current_device()} (the library runs on the current device)")


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def _weights(wq, w_scale, w_zero, N: int, K: int, device):
    _arg(wq, torch.uint8, (N, K // 2), "wq", device)
    _arg(w_scale, torch.float16, (N, K // 64), "w_scale", device)
    _arg(w_zero, torch.float16, (N, K // 64), "w_zero", device)


def _ws(ws, need: int, device, stream=None):
    """The caller's workspace (any dtype: its size in bytes is what the library is told), or
    a temporary one.  A temporary is dropped when the call returns, while the library's work
    on it is still queued on `stream`; the caching allocator is told about that stream
    (record_stream), so it does not hand the block to other work before that work is done
    (it otherwise tracks only the current stream, on which the block was allocated)."""
    if ws is None:
        t = workspace(need, device)
        if stream is not None:
            t.record_stream(stream)
        return t
    _arg(ws, None, None, "ws", device)
    return ws


def linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4a8_linear_workspace_bytes(M, N, K))


def prefill_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4a8_prefill_workspace_bytes(M, N, K))


def debug_workspace_bytes(m_cnt: int, n_cnt: int, K: int) -> int:
    return int(load().w4a8_debug_workspace_bytes(m_cnt, n_cnt, K))


_SIZE_REJECTED = (1 << 64) - 1   # what a size query returns for a shape the library rejects


def workspace(nbytes: int, device) -> torch.Tensor:
    """A caller-owned workspace buffer (uint8, at least 16-byte aligned).  For a rejected
    shape (size query = SIZE_MAX) a minimal buffer stands in: every call checks the shape
    before the workspace, so it then returns W4A8_ERR_SHAPE."""
    n = 16 if int(nbytes) == _SIZE_REJECTED else max(int(nbytes), 16)
    return torch.empty(n, dtype=torch.uint8, device=device)


def quant_pack(x: torch.Tensor, a_q=None, a_scale=None, rowsum=None, stream=None):
    """w4a8_quant_pack: x fp32 [M,K] -> (a_q int8 [M,K], s_a fp32 [M], rowsum int32 [M,K/64])."""
    _want(x, torch.float32, "x")
    M, K = x.shape
    dev = x.device
    a_q = torch.empty((M, K), dtype=torch.int8, device=dev) if a_q is None else a_q
    a_scale = torch.empty((M,), dtype=torch.float32, device=dev) if a_scale is None else a_scale
    rowsum = torch.empty((M, K // 64), dtype=torch.int32, device=dev) if rowsum is None else rowsum
    _arg(a_q, torch.int8, (M, K), "a_q", dev)
    _arg(a_scale, torch.float32, (M,), "a_scale", dev)
    _arg(rowsum, torch.int32, (M, K // 64), "rowsum", dev)
    rc = load().w4a8_quant_pack(_ptr(x), M, K, _ptr(a_q), _ptr(a_scale), _ptr(rowsum), _stream(stream))
    _check(rc, "w4a8_quant_pack")
    return a_q, a_scale, rowsum


def _quantized(a_q, a_scale, rowsum):
    """Shape (M, K) of a pre-quantized activation triple, after checking all three."""
    _want(a_q, torch.int8, "a_q")
    M, K = a_q.shape
    _arg(a_scale, torch.float32, (M,), "a_scale", a_q.device)
    _arg(rowsum, torch.int32, (M, K // 64), "rowsum", a_q.device)
    return M, K


def linear(a_q, a_scale, rowsum, wq, w_scale, w_zero, bias=None, y=None, ws=None, stream=None):
    """w4a8_linear: pre-quantized activations -> y fp32 [M,N]."""
    M, K = _quantized(a_q, a_scale, rowsum)
    dev = a_q.device
    N = _rows(wq)
    _weights(wq, w_scale, w_zero, N, K, dev)
    _arg(bias, torch.float32, (N,), "bias", dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev) if y is None else y
    _arg(y, torch.float32, (M, N), "y", dev)
    ws = _ws(ws, linear_workspace_bytes(M, N, K), dev, stream)
    rc = load().w4a8_linear(_ptr(a_q), _ptr(a_scale), _ptr(rowsum), _ptr(wq), _ptr(w_scale), _ptr(w_zero),
                            _ptr(bias), _ptr(y), M, N, K, _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "w4a8_linear")
    return y


def _rows(wq) -> int:
    _want(wq, torch.uint8, "wq")
    if wq.dim() != 2:
        raise ValueError(f"wq must be 2-D [N, K/2], got shape {tuple(wq.shape)}")
    return wq.shape[0]


def _prefill_args(x, wq, w_scale, w_zero, bias):
    """Shape (M, N, K) of a fused call, after checking x, the weights and the bias."""
    _want(x, torch.float32, "x")
    if x.dim() != 2:
        raise ValueError(f"x must be 2-D [M, K], got shape {tuple(x.shape)}")
    M, K = x.shape
    N = _rows(wq)
    _weights(wq, w_scale, w_zero, N, K, x.device)
    _arg(bias, torch.float32, (N,), "bias", x.device)
    return M, N, K


def prefill_linear(x, wq, w_scale, w_zero, bias=None, y=None, ws=None, stream=None):
    """w4a8_prefill_linear: fp32 x [M,K] -> y fp32 [M,N] (pre-pass + linear)."""
    M, N, K = _prefill_args(x, wq, w_scale, w_zero, bias)
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if y is None else y
    _arg(y, torch.float32, (M, N), "y", x.device)
    ws = _ws(ws, prefill_workspace_bytes(M, N, K), x.device, stream)
    rc = load().w4a8_prefill_linear(_ptr(x), _ptr(wq), _ptr(w_scale), _ptr(w_zero), _ptr(bias), _ptr(y),
                                    M, N, K, _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "w4a8_prefill_linear")
    return y


class LinearRef(ctypes.Structure):
    """w4a8_linear_ref: one entry of w4a8_prefill_linear_batch."""
    _fields_ = [("x", _P), ("wq", _P), ("w_scale", _P), ("w_zero", _P), ("bias", _P), ("y", _P),
                ("N", _I64), ("K", _I64), ("workspace", _P), ("workspace_bytes", _SZ)]


class Batch:
    """The entries of a w4a8_prefill_linear_batch call, checked and marshalled once: a sequence
    of dicts with x, wq, s_w, z_w, optional bias, y and ws (y and ws allocated when absent),
    one M for all.  `run(stream)` makes the call; `ys` are the outputs.  The tensors are held
    for the life of the object."""

    def __init__(self, entries, stream=None):
        entries = list(entries)
        self.count = len(entries)
        self.refs = (LinearRef * max(1, self.count))()
        self.keep, self.ys = [], []
        self.M = 0
        for i, e in enumerate(entries):
            x, wq, sw, zw, bias = e["x"], e["wq"], e["s_w"], e["z_w"], e.get("bias")
            m, N, K = _prefill_args(x, wq, sw, zw, bias)
            if i == 0:
                self.M = m
            elif m != self.M:
                raise ValueError(f"entry {i}: x has {m} rows, the batch {self.M}")
            y = e.get("y")
            y = torch.empty((m, N), dtype=torch.float32, device=x.device) if y is None else y
            _arg(y, torch.float32, (m, N), "y", x.device)
            ws = _ws(e.get("ws"), prefill_workspace_bytes(m, N, K), x.device, stream)
            self.refs[i] = LinearRef(x.data_ptr(), wq.data_ptr(), sw.data_ptr(), zw.data_ptr(),
                                     None if bias is None else bias.data_ptr(), y.data_ptr(), N, K, ws.data_ptr(),
                                     _nbytes(ws))
            self.keep += [x, wq, sw, zw, bias, ws]
            self.ys.append(y)

    def run(self, stream=None):
        rc = load().w4a8_prefill_linear_batch(ctypes.cast(self.refs, _P), self.count, self.M, _stream(stream))
        _check(rc, "w4a8_prefill_linear_batch")
        return self.ys


def prefill_linear_batch(entries, stream=None):
    """w4a8_prefill_linear_batch: the fused call on each entry in order (see Batch).  Returns
    the list of y."""
    return Batch(entries, stream).run(stream)


def prefill_linear_noalloc(x, wq, w_scale, w_zero, bias=None, y=None, stream=None):
    """w4a8_prefill_linear_noalloc: the fused call on the library's static scratch buffer,
    for callers that cannot allocate device memory.  Serialize calls that could overlap."""
    M, N, K = _prefill_args(x, wq, w_scale, w_zero, bias)
    y = torch.empty((M, N), dtype=torch.float32, device=x.device) if y is None else y
    _arg(y, torch.float32, (M, N), "y", x.device)
    rc = load().w4a8_prefill_linear_noalloc(_ptr(x), _ptr(wq), _ptr(w_scale), _ptr(w_zero), _ptr(bias), _ptr(y),
                                            M, N, K, _stream(stream))
    _check(rc, "w4a8_prefill_linear_noalloc")
    return y


def prefill_host_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4a8_prefill_host_workspace_bytes(M, N, K))


def _host(t, dtype, shape, name: str):
    """A host-buffer argument: a page-locked, contiguous CPU tensor of the C layout."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor, got {type(t).__name__}")
    # an empty tensor has no storage to pin; the library reads no pointer of an empty problem
    if t.device.type != "cpu" or (t.numel() and not t.is_pinned()):
        raise TypeError(f"{name} must be a page-locked host tensor (tensor.pin_memory())")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def prefill_linear_host(x, wq, w_scale, w_zero, bias=None, y=None, ws=None, stream=None):
    """w4a8_prefill_linear_host: page-locked host x fp32 [M,K] -> page-locked host y fp32
    [M,N]; the copies overlap the computation.  Asynchronous like every call: synchronize
    the stream before reading y."""
    _host(x, torch.float32, None, "x")
    if x.dim() != 2:
        raise ValueError(f"x must be 2-D [M, K], got shape {tuple(x.shape)}")
    M, K = x.shape
    N = _rows(wq)
    dev = wq.device
    _weights(wq, w_scale, w_zero, N, K, dev)
    _arg(bias, torch.float32, (N,), "bias", dev)
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32)
        y = y.pin_memory() if y.numel() else y
    _host(y, torch.float32, (M, N), "y")
    ws = _ws(ws, prefill_host_workspace_bytes(M, N, K), dev, stream)
    rc = load().w4a8_prefill_linear_host(_ptr(x), _ptr(wq), _ptr(w_scale), _ptr(w_zero), _ptr(bias), _ptr(y),
                                         M, N, K, _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "w4a8_prefill_linear_host")
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
    _arg(act, None, None, "act", x.device)
    rc = load().w4a8_prepare_activations(_ptr(x), M, K, _ptr(act), _nbytes(act), _stream(stream))
    _check(rc, "w4a8_prepare_activations")
    return act


def prepare_weights(wq, w_scale, w_zero, pw=None, stream=None):
    """w4a8_prepare_weights: the tensor-core weight operand and the scale / zero layout
    (an opaque buffer, returned)."""
    N = _rows(wq)
    K = 2 * wq.shape[1]
    _weights(wq, w_scale, w_zero, N, K, wq.device)
    pw = workspace(prepared_weights_bytes(N, K), wq.device) if pw is None else pw
    _arg(pw, None, None, "pw", wq.device)
    rc = load().w4a8_prepare_weights(_ptr(wq), _ptr(w_scale), _ptr(w_zero), N, K, _ptr(pw), _nbytes(pw),
                                     _stream(stream))
    _check(rc, "w4a8_prepare_weights")
    return pw


def _out(y, shape, device, out_dtype):
    dt = torch.float32 if out_dtype is None else out_dtype
    if dt not in _OUT_DTYPES:
        raise TypeError(f"y: unsupported output dtype {dt}")
    y = torch.empty(shape, dtype=dt, device=device) if y is None else y
    _arg(y, dt, shape, "y", device)
    return y, _OUT_DTYPES[dt]


def prefill_linear_ex(x, wq, w_scale, w_zero, bias=None, y=None, out_dtype=None, clamp=(-math.inf, math.inf),
                      ws=None, stream=None):
    """w4a8_prefill_linear_ex: the fused call with the epilogue clamp and an fp32 or bf16 y."""
    M, N, K = _prefill_args(x, wq, w_scale, w_zero, bias)
    y, code = _out(y, (M, N), x.device, out_dtype if y is None else y.dtype)
    ws = _ws(ws, prefill_workspace_bytes(M, N, K), x.device, stream)
    rc = load().w4a8_prefill_linear_ex(_ptr(x), _ptr(wq), _ptr(w_scale), _ptr(w_zero), _ptr(bias), _ptr(y), code,
                                       float(clamp[0]), float(clamp[1]), M, N, K, _ptr(ws), _nbytes(ws),
                                       _stream(stream))
    _check(rc, "w4a8_prefill_linear_ex")
    return y


def linear_ex(a_q, a_scale, rowsum, wq, w_scale, w_zero, bias=None, y=None, out_dtype=None,
              clamp=(-math.inf, math.inf), ws=None, stream=None):
    """w4a8_linear_ex: pre-quantized activations, epilogue clamp, fp32 or bf16 y."""
    M, K = _quantized(a_q, a_scale, rowsum)
    dev = a_q.device
    N = _rows(wq)
    _weights(wq, w_scale, w_zero, N, K, dev)
    _arg(bias, torch.float32, (N,), "bias", dev)
    y, code = _out(y, (M, N), dev, out_dtype if y is None else y.dtype)
    ws = _ws(ws, linear_workspace_bytes(M, N, K), dev, stream)
    rc = load().w4a8_linear_ex(_ptr(a_q), _ptr(a_scale), _ptr(rowsum), _ptr(wq), _ptr(w_scale), _ptr(w_zero),
                               _ptr(bias), _ptr(y), code, float(clamp[0]), float(clamp[1]), M, N, K, _ptr(ws),
                               _nbytes(ws), _stream(stream))
    _check(rc, "w4a8_linear_ex")
    return y


def _prepared(act, pw, bias, M: int, N: int, K: int):
    """Check the opaque operands of a prepared call against the sizes the library derives
    from (M, N, K): the C call takes no buffer lengths, so this is the only check."""
    _want(act, None, "act")
    dev = act.device
    if min(M, N, K) < 0:
        raise ValueError(f"negative size in (M, N, K) = {(M, N, K)}")
    if M and N and K > 0 and K % 64 == 0:
        _arg(act, None, None, "act", dev, min_bytes=prepared_activations_bytes(M, K))
        _arg(pw, None, None, "pw", dev, min_bytes=prepared_weights_bytes(N, K))
    else:
        _arg(pw, None, None, "pw", dev)
    _arg(bias, torch.float32, (N,), "bias", dev)
    return dev


def linear_prepared_ex(act, pw, M: int, N: int, K: int, bias=None, y=None, out_dtype=None,
                       clamp=(-math.inf, math.inf), stream=None):
    """w4a8_linear_prepared_ex: prepared operands, epilogue clamp, fp32 or bf16 y."""
    dev = _prepared(act, pw, bias, M, N, K)
    y, code = _out(y, (M, N), dev, out_dtype if y is None else y.dtype)
    rc = load().w4a8_linear_prepared_ex(_ptr(act), _ptr(pw), _ptr(bias), _ptr(y), code, float(clamp[0]),
                                        float(clamp[1]), M, N, K, _stream(stream))
    _check(rc, "w4a8_linear_prepared_ex")
    return y


def linear_prepared(act, pw, M: int, N: int, K: int, bias=None, y=None, stream=None):
    """w4a8_linear_prepared: contraction + epilogue from prepared operands -> y fp32 [M,N]."""
    dev = _prepared(act, pw, bias, M, N, K)
    y = torch.empty((M, N), dtype=torch.float32, device=dev) if y is None else y
    _arg(y, torch.float32, (M, N), "y", dev)
    rc = load().w4a8_linear_prepared(_ptr(act), _ptr(pw), _ptr(bias), _ptr(y), M, N, K, _stream(stream))
    _check(rc, "w4a8_linear_prepared")
    return y


def linear_act_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().w4a8_linear_act_workspace_bytes(M, N, K))


def linear_act(act, wq, w_scale, w_zero, M: int, N: int, K: int, bias=None, y=None, ws=None, stream=None):
    """w4a8_linear_act: contraction + epilogue from prepared activations and the packed
    weights as given -> y fp32 [M,N]."""
    _want(act, None, "act")
    dev = act.device
    if min(M, N, K) < 0:
        raise ValueError(f"negative size in (M, N, K) = {(M, N, K)}")
    if M and N and K > 0 and K % 64 == 0:
        _arg(act, None, None, "act", dev, min_bytes=prepared_activations_bytes(M, K))
    _weights(wq, w_scale, w_zero, N, K, dev)
    _arg(bias, torch.float32, (N,), "bias", dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev) if y is None else y
    _arg(y, torch.float32, (M, N), "y", dev)
    ws = _ws(ws, linear_act_workspace_bytes(M, N, K), dev, stream)
    rc = load().w4a8_linear_act(_ptr(act), _ptr(wq), _ptr(w_scale), _ptr(w_zero), _ptr(bias), _ptr(y), M, N, K,
                                _ptr(ws), _nbytes(ws), _stream(stream))
    _check(rc, "w4a8_linear_act")
    return y


def debug_block_acc(a_q, wq, N, m0=0, m_cnt=None, n0=0, n_cnt=None, ws=None, stream=None):
    """w4a8_debug_block_acc: exact per-block int32 accumulators [m_cnt, n_cnt, K/64]."""
    _want(a_q, torch.int8, "a_q")
    M, K = a_q.shape
    _arg(wq, torch.uint8, (N, K // 2), "wq", a_q.device)
    m_cnt = M - m0 if m_cnt is None else m_cnt
    n_cnt = N - n0 if n_cnt is None else n_cnt
    if not (0 <= m0 and 0 <= m_cnt and m0 + m_cnt <= M and 0 <= n0 and 0 <= n_cnt and n0 + n_cnt <= N):
        raise ValueError(f"window rows [{m0}, {m0}+{m_cnt}) x cols [{n0}, {n0}+{n_cnt}) outside [{M}] x [{N}]")
    acc = torch.empty((m_cnt, n_cnt, K // 64), dtype=torch.int32, device=a_q.device)
    ws = _ws(ws, debug_workspace_bytes(m_cnt, n_cnt, K), a_q.device, stream)
    rc = load().w4a8_debug_block_acc(_ptr(a_q), _ptr(wq), M, N, K, m0, m_cnt, n0, n_cnt, _ptr(acc),
                                     _ptr(ws), _nbytes(ws), _stream(stream))
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

    def kernels(self) -> int:
        """Kernel launches per replay (w4a8_tape_kernels)."""
        if self.handle is None:
            raise RuntimeError("tape not recorded")
        return int(load().w4a8_tape_kernels(self.handle))

    def free(self):
        if self.handle is not None:
            load().w4a8_tape_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

