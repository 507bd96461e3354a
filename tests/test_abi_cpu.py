"""The C-ABI library loads and exports every symbol include/w4a8.h declares; argument
validation that needs no GPU (shapes, null pointers, workspace sizes) returns the
documented status codes.  No compute call is made here."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a8.h")


@pytest.fixture(scope="module")
def lib():
    from w4a8_block_quantized_gb300 import build, binding
    build.build()
    return binding.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a8_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    syms = declared_symbols()
    for need in ("w4a8_quant_pack", "w4a8_linear", "w4a8_prefill_linear", "w4a8_debug_block_acc"):
        assert need in syms


def test_every_declared_symbol_is_exported(lib):
    from w4a8_block_quantized_gb300 import binding
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in binding.SIGNATURES, f"binding lacks {name}"


def test_status_strings(lib):
    from w4a8_block_quantized_gb300 import binding as b
    for code in (b.W4A8_OK, b.W4A8_ERR_ARG, b.W4A8_ERR_ALIGN, b.W4A8_ERR_SHAPE, b.W4A8_ERR_CUDA,
                 b.W4A8_ERR_TIMEOUT, b.W4A8_ERR_WORKSPACE, b.W4A8_ERR_DEVICE):
        s = b.status_string(code)
        assert s and s != "unknown status"
    assert b.status_string(12345) == "unknown status"
    assert lib.w4a8_abi_version() == 204


def test_shape_checks_need_no_gpu(lib):
    from w4a8_block_quantized_gb300 import binding as b
    P = ctypes.c_void_p
    dummy = P(16)  # never dereferenced: validation fails first
    assert lib.w4a8_quant_pack(dummy, 4, 100, dummy, dummy, dummy, None) == b.W4A8_ERR_SHAPE
    assert lib.w4a8_quant_pack(dummy, 4, 0, dummy, dummy, dummy, None) == b.W4A8_ERR_SHAPE
    assert lib.w4a8_quant_pack(dummy, -1, 64, dummy, dummy, dummy, None) == b.W4A8_ERR_ARG
    assert lib.w4a8_quant_pack(None, 4, 64, dummy, dummy, dummy, None) == b.W4A8_ERR_ARG
    assert lib.w4a8_quant_pack(P(8), 4, 64, dummy, dummy, dummy, None) == b.W4A8_ERR_ALIGN
    # empty problems are valid no-ops
    assert lib.w4a8_quant_pack(None, 0, 64, None, None, None, None) == b.W4A8_OK
    assert lib.w4a8_prefill_linear(None, None, None, None, None, None, 0, 8, 64, None, 0, None) == b.W4A8_OK
    assert lib.w4a8_linear(None, None, None, None, None, None, None, None, 8, 0, 64, None, 0, None) == b.W4A8_OK
    assert lib.w4a8_linear(dummy, dummy, dummy, dummy, dummy, dummy, None, dummy, 8, 8, 96, dummy, 1 << 20,
                           None) == b.W4A8_ERR_SHAPE
    # workspace too small is reported before any launch
    # (the tensor-core form, and the few-token form after a separate pre-pass)
    for M, N, K in ((16, 8, 64), (8, 8, 4096)):
        need = lib.w4a8_prefill_workspace_bytes(M, N, K)
        assert need > 0
        assert lib.w4a8_prefill_linear(dummy, dummy, P(32), P(32), None, dummy, M, N, K, dummy, need - 1,
                                       None) == b.W4A8_ERR_WORKSPACE
    # debug window outside the problem
    assert lib.w4a8_debug_block_acc(dummy, dummy, 8, 8, 64, 4, 8, 0, 8, dummy, dummy, 1 << 20,
                                    None) == b.W4A8_ERR_SHAPE


def test_workspace_sizes(lib):
    # operand planes (2 bytes per activation) + row-sum entries (16 bytes per token and block)
    # + expanded weights (1 byte each) + scales and weight-side zero-point rows (4 + 16 bytes)
    for M in (512, 4096):
        N, K = 3072, 1024
        nb = K // 64
        lin = lib.w4a8_linear_workspace_bytes(M, N, K)
        pre = lib.w4a8_prefill_workspace_bytes(M, N, K)
        assert lin >= 2 * M * K + nb * M * 16 + N * K + nb * N * 20
        assert pre >= lin + 4 * M
    # w4a8_linear_act: below 4096 tokens the contraction reads the packed weights itself (no
    # workspace); from 4096 on the weight records go into the workspace
    assert lib.w4a8_linear_act_workspace_bytes(512, 3072, 1024) == 0
    assert lib.w4a8_linear_act_workspace_bytes(4096, 3072, 1024) == lib.w4a8_prepared_weights_bytes(3072, 1024)
    assert lib.w4a8_linear_workspace_bytes(0, N, K) == 0
    assert lib.w4a8_linear_workspace_bytes(M, N, 100) == ctypes.c_size_t(-1).value
    assert lib.w4a8_debug_workspace_bytes(7, 9, 128) >= 7 * 256 + 9 * 128


def test_few_token_workspace_sizes(lib):
    """Up to W4A8_DECODE_MAX_M tokens the linear needs no scratch; the fused call none when
    the kernel quantizes the rows itself (M * K <= 16384), else the pre-pass outputs in the
    API layout; one token more switches to the tensor-core form."""
    N = 3072
    for M in range(1, 9):
        for K in (1024, 2048, 4096, 16384):
            nb = K // 64
            assert lib.w4a8_linear_workspace_bytes(M, N, K) == 0
            pre = lib.w4a8_prefill_workspace_bytes(M, N, K)
            if M * K <= 16384:
                assert pre == 0
            else:
                assert M * K + 4 * M + 4 * M * nb <= pre <= M * K + 4 * M + 4 * M * nb + 3 * 256
    assert lib.w4a8_linear_workspace_bytes(9, N, 1024) >= N * 1024
    assert lib.w4a8_prefill_workspace_bytes(9, N, 1024) >= N * 1024


def test_epilogue_arguments_rejected_before_launch(lib):
    """The *_ex calls reject an unknown output type and clamp bounds with lo > hi or a NaN
    before touching the device."""
    import math
    from w4a8_block_quantized_gb300 import binding as b
    d = ctypes.c_void_p(1 << 20)
    for dt, lo, hi in ((2, -1.0, 1.0), (-1, -1.0, 1.0), (0, 1.0, -1.0), (1, math.nan, 1.0), (0, -1.0, math.nan)):
        assert lib.w4a8_prefill_linear_ex(d, d, d, d, None, d, dt, lo, hi, 4, 8, 64, None, 0, None) == b.W4A8_ERR_ARG
        assert lib.w4a8_linear_ex(d, d, d, d, d, d, None, d, dt, lo, hi, 4, 8, 64, None, 0, None) == b.W4A8_ERR_ARG
        assert lib.w4a8_linear_prepared_ex(d, d, None, d, dt, lo, hi, 4, 8, 64, None) == b.W4A8_ERR_ARG


def test_tape_arguments_rejected(lib):
    from w4a8_block_quantized_gb300 import binding as b
    assert lib.w4a8_tape_begin(None) == b.W4A8_ERR_ARG            # the default stream is not captured
    h = ctypes.c_void_p()
    assert lib.w4a8_tape_end(None, ctypes.byref(h)) == b.W4A8_ERR_ARG
    assert lib.w4a8_tape_end(ctypes.c_void_p(1 << 20), None) == b.W4A8_ERR_ARG
    assert lib.w4a8_tape_replay(None, None) == b.W4A8_ERR_ARG
    lib.w4a8_tape_free(None)                                      # a no-op
    assert lib.w4a8_tape_kernels(None) == -1


def test_deep_few_token_rows_take_the_tensor_core_form(lib):
    """Eight tokens of K = 32768 do not fit the few-token kernel's shared memory: the linear
    then needs the tensor-core form's workspace; K = 16384 still fits."""
    assert lib.w4a8_linear_workspace_bytes(8, 256, 16384) == 0
    assert lib.w4a8_linear_workspace_bytes(8, 256, 32768) > 0
    assert lib.w4a8_linear_workspace_bytes(1, 256, 32768) == 0


class _named:
    """Adds the call's name to an assertion raised inside the block."""

    def __init__(self, name):
        self.name = name

    def __enter__(self):
        return self

    def __exit__(self, et, e, tb):
        if et is AssertionError:
            raise AssertionError(f"{self.name}: {e}") from e
        return False


def test_binding_rejects_host_tensors_before_the_library():
    """No binding call hands a host address to the library: a CPU tensor anywhere in the
    argument list raises TypeError in the binding, before any entry point runs."""
    import torch
    from w4a8_block_quantized_gb300 import binding as b

    M, N, K = 4, 8, 64
    x = torch.zeros((M, K))
    a_q = torch.zeros((M, K), dtype=torch.int8)
    s_a = torch.zeros(M)
    rs = torch.zeros((M, 1), dtype=torch.int32)
    wq = torch.zeros((N, K // 2), dtype=torch.uint8)
    sw = torch.zeros((N, 1), dtype=torch.float16)
    buf = torch.zeros(1 << 16, dtype=torch.uint8)
    calls = {
        "quant_pack": lambda: b.quant_pack(x),
        "linear": lambda: b.linear(a_q, s_a, rs, wq, sw, sw),
        "linear_ex": lambda: b.linear_ex(a_q, s_a, rs, wq, sw, sw),
        "prefill_linear": lambda: b.prefill_linear(x, wq, sw, sw),
        "prefill_linear_ex": lambda: b.prefill_linear_ex(x, wq, sw, sw),
        "prefill_linear_noalloc": lambda: b.prefill_linear_noalloc(x, wq, sw, sw),
        "prepare_activations": lambda: b.prepare_activations(x),
        "prepare_weights": lambda: b.prepare_weights(wq, sw, sw),
        "linear_prepared": lambda: b.linear_prepared(buf, buf, M, N, K),
        "linear_prepared_ex": lambda: b.linear_prepared_ex(buf, buf, M, N, K),
        "debug_block_acc": lambda: b.debug_block_acc(a_q, wq, N),
    }
    for name, call in calls.items():
        with pytest.raises(TypeError, match="CUDA tensor"), _named(name):
            call()
    with pytest.raises(TypeError, match="torch.Tensor"):
        b._arg(object(), None, None, "y")


def _align(v):
    return (v + 255) & ~255


def test_host_call_workspace_and_chunking(lib):
    """The host-buffer call's workspace: the device copies of x and y, then either the fused
    call's scratch (one chunk) or the prepared weights and one prepared-activation buffer per
    compute stream (at most four), sized for the largest chunk.  A call is cut into at most
    sixteen chunks of whole token tiles, each moving at least 8 MiB of x and y; the tiles are
    spread evenly, so the first (tiles mod chunks) chunks take one tile more than the rest.
    Chunks are 128-token tiles below 4096 rows; a one-chunk call needs the fused call's
    scratch, which covers either token-tile width."""
    def plan(M, N, K, tw):
        chunks = 1 if M <= 8 else max(1, min(16, M // tw, M * (K + N) * 4 // (8 << 20)))
        tiles = -(-M // tw)
        largest = min((tiles // chunks + (tiles % chunks > 0)) * tw, M)
        return chunks, largest

    def base(M, N, K):
        return _align(_align(M * K * 4) + M * N * 4)

    def act_bytes(rows, K, tw):  # token records of width tw, then the row scales
        return _align(-(-rows // tw) * (K // 64) * 144 * tw) + _align(rows * 4)

    def want(M, N, K, tw):
        chunks, last = plan(M, N, K, tw)
        if chunks == 1:
            return base(M, N, K) + lib.w4a8_prefill_workspace_bytes(M, N, K)
        return base(M, N, K) + lib.w4a8_prepared_weights_bytes(N, K) + min(chunks, 4) * act_bytes(last, K, tw)

    cases = [  # (M, N, K, chunks, rows of the largest chunk) with 128-token tiles
        (512, 3072, 1024, 1, 512),        # the pp512 linear: 8 MiB in all, one chunk
        (700, 200, 256, 1, 700),
        (3, 256, 1024, 1, 3),
        (1500, 2560, 1024, 2, 768),       # 12 tiles: 6 + 6 (the second ragged)
        (2048, 4096, 1024, 5, 512),       # 16 tiles: 4 + 3 + 3 + 3 + 3
        (1000, 8192, 1024, 4, 256),       # 8 tiles: 2 each
        (2048, 4096, 2048, 6, 384),       # 16 tiles: 3 3 3 3 2 2
    ]
    for M, N, K, chunks, last in cases:
        assert plan(M, N, K, 128) == (chunks, last), (M, N, K)
        assert act_bytes(last, K, 128) == lib.w4a8_prepared_activations_bytes(last, K)
        got = lib.w4a8_prefill_host_workspace_bytes(M, N, K)
        assert got == want(M, N, K, 128), (M, N, K)
    # 256-token records: chunks of whole 256-row tiles, below 4096 rows each
    assert plan(8192, 14336, 4096, 256)[0] == 16 and plan(16384, 1024, 1024, 256) == (16, 1024)
    for M, N, K in ((8192, 14336, 4096), (8300, 512, 256), (9000, 1536, 512), (16384, 1024, 1024)):
        chunks, last = plan(M, N, K, 256)
        assert chunks > 1 and last < 4096
        got = lib.w4a8_prefill_host_workspace_bytes(M, N, K)
        assert got >= want(M, N, K, 256)
    assert lib.w4a8_prefill_host_workspace_bytes(0, 64, 128) == 0
    assert lib.w4a8_prefill_host_workspace_bytes(4, 64, 100) == ctypes.c_size_t(-1).value


def test_host_call_arguments_rejected_before_launch(lib):
    from w4a8_block_quantized_gb300 import binding as b
    P = ctypes.c_void_p
    d = P(1 << 20)
    M, N, K = 512, 64, 128
    need = lib.w4a8_prefill_host_workspace_bytes(M, N, K)
    assert lib.w4a8_prefill_linear_host(d, d, d, d, None, d, M, N, 96, d, need, None) == b.W4A8_ERR_SHAPE
    assert lib.w4a8_prefill_linear_host(None, d, d, d, None, d, M, N, K, d, need, None) == b.W4A8_ERR_ARG
    assert lib.w4a8_prefill_linear_host(d, d, d, d, None, None, M, N, K, d, need, None) == b.W4A8_ERR_ARG
    assert lib.w4a8_prefill_linear_host(d, d, d, d, None, d, M, N, K, None, need, None) == b.W4A8_ERR_ARG
    assert lib.w4a8_prefill_linear_host(d, d, d, d, None, d, M, N, K, P((1 << 20) + 8), need, None) == \
        b.W4A8_ERR_ALIGN
    assert lib.w4a8_prefill_linear_host(d, d, d, d, None, d, M, N, K, d, need - 1, None) == b.W4A8_ERR_WORKSPACE
    assert lib.w4a8_prefill_linear_host(None, None, None, None, None, None, 0, N, K, None, 0, None) == b.W4A8_OK


def test_binding_host_call_wants_page_locked_buffers():
    import torch
    from w4a8_block_quantized_gb300 import binding as b
    x = torch.zeros((4, 64))
    wq = torch.zeros((8, 32), dtype=torch.uint8)
    sw = torch.zeros((8, 1), dtype=torch.float16)
    with pytest.raises(TypeError, match="page-locked"):
        b.prefill_linear_host(x, wq, sw, sw)
    # an empty problem has nothing to pin: its host tensors pass the check
    b._host(torch.empty((0, 64)), torch.float32, (0, 64), "x")
    with pytest.raises(TypeError, match="page-locked"):
        b._host(torch.empty((1, 64)), torch.float32, (1, 64), "x")


def test_plain_c_client(lib, tmp_path):
    """The header compiles as strict C99 and a C program links against the library and gets
    the documented answers from the calls that need no GPU."""
    import subprocess
    from w4a8_block_quantized_gb300 import binding
    libdir = os.path.dirname(binding.LIB_PATH)
    exe = tmp_path / "c_client"
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_client.c"),
                    "-L", libdir, "-lw4a8", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr
