"""TEST INFRASTRUCTURE ONLY: ctypes loader for the plain C oracle in ``w4a8_oracle.c``.

The oracle is the slow CPU statement of the W4A8 block-64 quantized linear
("MNN LLM inference on the SpacemiT K3", section 3 eqs. (1)-(3) and section 4).
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and this
package imports nothing from the product package.

Arrays cross the boundary as numpy arrays; fp16 inputs travel as their raw
16-bit patterns and are decoded by the C file itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w4a8_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict[str, ctypes.CDLL] = {}

BLOCK = 64


def build(defines: tuple[str, ...] = (), tag: str = "oracle", openmp: bool = True) -> str:
    """Compile the oracle into ``oracle/_build/lib<tag>.so`` and return its path.

    ``defines`` are extra ``-D`` macros (the mutation tests use them to compile
    deliberately broken copies).  Rebuilds only when the source is newer.
    """
    os.makedirs(_BUILD, exist_ok=True)
    out = os.path.join(_BUILD, f"lib{tag}.so")
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra"]
    cmd.append("-fopenmp" if openmp else "-Wno-unknown-pragmas")
    cmd += [f"-D{d}" for d in defines]
    tmp = out + f".tmp{os.getpid()}"
    cmd += [_SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def lib(tag: str = "oracle", defines: tuple[str, ...] = ()) -> ctypes.CDLL:
    with _LOCK:
        if tag not in _LIBS:
            path = build(defines=defines, tag=tag)
            cdll = ctypes.CDLL(path)
            _declare(cdll)
            _LIBS[tag] = cdll
        return _LIBS[tag]


def _declare(c: ctypes.CDLL) -> None:
    P = ctypes.c_void_p
    L = ctypes.c_long
    c.oracle_half_to_double.restype = ctypes.c_double
    c.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    c.oracle_quant_pack.restype = None
    c.oracle_quant_pack.argtypes = [P, L, L, P, P, P]
    for name in ("oracle_block_acc", "oracle_block_acc_nibble"):
        f = getattr(c, name)
        f.restype = None
        f.argtypes = [P, P, L, L, L, L, L, L, L, P]
    c.oracle_linear_rows.restype = None
    c.oracle_linear_rows.argtypes = [P, P, P, P, P, P, P, L, L, L, P, L, P, P]
    c.oracle_prefill_linear_rows.restype = None
    c.oracle_prefill_linear_rows.argtypes = [P, P, P, P, P, L, L, L, P, L, P, P, P, P, P]
    c.oracle_num_threads.restype = ctypes.c_int
    c.oracle_num_threads.argtypes = []


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _bits16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    return _c(a, np.uint16)


def half_to_double(bits, tag: str = "oracle") -> np.ndarray:
    """Decode raw fp16 bit patterns with the oracle's own routine."""
    c = lib(tag)
    flat = _bits16(bits).ravel()
    return np.array([c.oracle_half_to_double(int(h)) for h in flat]).reshape(np.shape(bits))


def quant_pack(x, tag: str = "oracle"):
    """Section 4 step 1: returns (a_q int8 [M,K], s_a fp32 [M], rs int32 [M,K/64])."""
    x = _c(x, np.float32)
    M, K = x.shape
    a_q = np.empty((M, K), np.int8)
    s_a = np.empty((M,), np.float32)
    rs = np.empty((M, K // BLOCK), np.int32)
    lib(tag).oracle_quant_pack(_p(x), M, K, _p(a_q), _p(s_a), _p(rs))
    return a_q, s_a, rs


def block_acc(a_q, wq, N, m0=0, mc=None, n0=0, nc=None, nibble=False, tag: str = "oracle"):
    """Per-block int32 accumulators acc[mc, nc, K/64] for a window (section 3 eq. (2))."""
    a_q = _c(a_q, np.int8)
    wq = _c(wq, np.uint8)
    M, K = a_q.shape
    mc = M - m0 if mc is None else mc
    nc = N - n0 if nc is None else nc
    acc = np.empty((mc, nc, K // BLOCK), np.int32)
    f = lib(tag).oracle_block_acc_nibble if nibble else lib(tag).oracle_block_acc
    f(_p(a_q), _p(wq), M, N, K, m0, mc, n0, nc, _p(acc))
    return acc


def linear(a_q, s_a, rs, wq, s_w, z_w, bias=None, rows=None, tag: str = "oracle"):
    """fp64 output y and the tolerance magnitude sum_b |block term| for the given rows."""
    a_q = _c(a_q, np.int8)
    s_a = _c(s_a, np.float32)
    rs = _c(rs, np.int32)
    wq = _c(wq, np.uint8)
    sw = _bits16(s_w)
    zw = _bits16(z_w)
    b = None if bias is None else _c(bias, np.float32)
    M, K = a_q.shape
    N = sw.shape[0]
    r = None if rows is None else _c(rows, np.int64)
    n_rows = M if r is None else len(r)
    y = np.empty((n_rows, N), np.float64)
    bound = np.empty((n_rows, N), np.float64)
    lib(tag).oracle_linear_rows(_p(a_q), _p(s_a), _p(rs), _p(wq), _p(sw), _p(zw), _p(b),
                                M, N, K, _p(r), n_rows, _p(y), _p(bound))
    return y, bound


def prefill_linear(x, wq, s_w, z_w, bias=None, rows=None, tag: str = "oracle"):
    """Whole prefill linear from fp32 x for the given rows.

    Returns (y fp64 [n_rows,N], bound [n_rows,N], a_q [n_rows,K], s_a [n_rows], rs [n_rows,K/64]).
    """
    x = _c(x, np.float32)
    wq = _c(wq, np.uint8)
    sw = _bits16(s_w)
    zw = _bits16(z_w)
    b = None if bias is None else _c(bias, np.float32)
    M, K = x.shape
    N = sw.shape[0]
    r = None if rows is None else _c(rows, np.int64)
    n_rows = M if r is None else len(r)
    a_q = np.empty((n_rows, K), np.int8)
    s_a = np.empty((n_rows,), np.float32)
    rs = np.empty((n_rows, K // BLOCK), np.int32)
    y = np.empty((n_rows, N), np.float64)
    bound = np.empty((n_rows, N), np.float64)
    lib(tag).oracle_prefill_linear_rows(_p(x), _p(wq), _p(sw), _p(zw), _p(b), M, N, K,
                                        _p(r), n_rows, _p(a_q), _p(s_a), _p(rs), _p(y), _p(bound))
    return y, bound, a_q, s_a, rs


def num_threads(tag: str = "oracle") -> int:
    return int(lib(tag).oracle_num_threads())


def bf16_round(v) -> np.ndarray:
    """Nearest value with an 8-bit significand (bfloat16: 1 implicit + 7 stored bits, the
    fp32 exponent range), ties to the even significand; returned as float64.  Written from
    the definition: v = f * 2^e with 1/2 <= |f| < 1, f * 2^8 rounded half-to-even, scaled
    back.  Below the normal range (|v| < 2^-126) the step is fixed at 2^-133."""
    v = np.asarray(v, dtype=np.float64)
    f, e = np.frexp(v)
    e = np.maximum(e, -125)                 # 2^-126 = 0.5 * 2^-125: subnormal step 2^-133
    out = np.rint(np.ldexp(v, 8 - e))       # np.rint rounds half to even
    return np.ldexp(out, e - 8)


def epilogue(y, clamp_lo=-np.inf, clamp_hi=np.inf, out_dtype: str = "f32") -> np.ndarray:
    """Section 4 step 3's store of the output: clamp to [clamp_lo, clamp_hi], then the
    value the output type holds (fp32: IEEE round to nearest even; bf16: bf16_round).
    y is the exact (fp64) result; returns float64."""
    v = np.clip(np.asarray(y, dtype=np.float64), clamp_lo, clamp_hi)
    if out_dtype == "f32":
        return v.astype(np.float32).astype(np.float64)
    if out_dtype == "bf16":
        return bf16_round(v)
    raise ValueError(out_dtype)
